// Fused SwiGLU expert for narrow experts (model width D <= 256): both expert
// GEMMs of a 128-row tile in one CTA, the activation kept on chip.  The
// "calculation" step of the MagiMoE operator library, with its fusion of
// steps to cut intermediate results and memory traffic ("Sand.ai: The
// world's first 100-billion-parameter open-source MoE video generation model
// MAGI Preview" (36kr), section "02. Two Key Technical Decision Points"),
// for the head-local experts of that section (one 256-dim head slice in and
// out).
//
// Per tile (128 rows of one expert group; its x rows, the head slices of the
// group's tokens, are copied from x by source token into shared memory and
// stay there for the whole tile) and per 128-column piece p of the
// intermediate:
//   1. acc1 = x W13[256p, 256p + 256)^T   (gate | up of chunk 2p, gate | up of
//      chunk 2p+1: 64 columns each, TMEM)
//   2. act_p = bf16(silu(gate) * up)       (epilogue -> shared memory, two
//      128-byte-swizzled 64-column sub-tiles)
//   3. acc2 += act_p W_down[:, 128p, 128p + 128)^T   (TMEM, D columns)
// and at the end y = bf16(acc2).  Every MMA is 128 x 256 x 16 (both the
// gate/up and the down products are 256 wide).  acc1 has one buffer (acc1
// 256 + acc2 256 columns fill tensor memory); the eight epilogue warps read
// it out quickly and the MMA thread issues piece p-1's down products in
// between, so the tensor pipe keeps running.  (A 128 x 128 x 16 MMA keeps
// the pipe's full rate too, but 64-column pieces with two gate/up
// accumulators, which that would allow, ran 25-35% slower: twice the
// SwiGLU hand-offs and gate/up MMAs per tile.)  act is
// rounded to bf16 exactly as the two separate GEMMs round it, and both
// products run the same MMA sequence, so y has the bits of the unfused pair.
//
// Work split: tiles are numbered group-major (a group's 128-row blocks
// consecutively, from a prefix table of the groups' tile counts) and handed
// out statically (tile = blockIdx + i * gridDim), so a group's blocks run on
// neighbouring CTAs at the same time and read its weights from DRAM once,
// the rest from L2.  (One CTA taking every block of a group in turn read
// each group's weights once per block: 148 groups' weights in flight do not
// stay in L2 between blocks.)  Roles (384 threads, one CTA per SM):
// warp 0 lane 0 loads w13 and W_down slices with TMA through a ring in the
// MMA thread's order, warp 1 lane 0 issues tcgen05.mma, warps 2..9 run
// SwiGLU and store y (warps w and w + 4 share TMEM lane quadrant w % 4; the
// first takes chunk 2p and the first half of y's columns, the second chunk
// 2p+1 and the rest), warps 10..11 gather the next tile's x rows with
// cp.async as soon as the gate/up products are done with the current ones
// (x is read from L2, 66 MB for the 10,752-token head-local workload, so
// the sorted copy x_perm never exists).  Every wait is bounded as in the
// GEMM engine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "internal.h"
#include "moe.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kFStages = 3;
constexpr int kFSub = kBM * kBK * 2;            // one 128-row x 64-column bf16 sub-tile: 16 KB
constexpr int kFStageBytes = 2 * kFSub;         // one 256-row x 64-column slice of w13 or W_down
constexpr int kFMaxD = 256;
constexpr int kFXBytes = (kFMaxD / kBK) * kFSub;  // the tile's x rows: 64 KB at D = 256
constexpr int kFActBytes = 2 * kFSub;           // one piece of act: two 64-column sub-tiles
constexpr int kFDynBytes = kFXBytes + kFStages * kFStageBytes + 2 * kFActBytes + 1024;
constexpr uint32_t kAcc2Col = 256;              // TMEM column of the down-projection accumulator
constexpr int kFEpiWarps = 8;
constexpr int kFGatherWarp = 2 + kFEpiWarps;  // the first warp after the epilogue warps
constexpr int kFGatherWarps = 2;
constexpr int kFThreads = 32 * (kFGatherWarp + kFGatherWarps);
constexpr int kFGatherRows = kBM / kFGatherWarps;  // tile rows per gather warp

struct FfnFusedArgs {
  const int* offsets;  // [groups + 1] group row offsets
  const int* tiles;    // [groups + 1] exclusive prefix of the groups' 128-row tile counts
  int groups;
  int rows;            // rows of y (the sorted rows of all groups)
  // Row r of a tile of group g is x[src[r], (g / head_groups) * D + (0 .. D)):
  // x is [T, x_ld] bf16, src [rows] token indices
  const uint16_t* x;
  int64_t x_ld;
  const int* src;
  int T;
  int head_groups;
  int D, I;
  uint16_t* y;         // [rows, D]
  int* status;
  uint64_t wait_ns;
  // Self-test only: the weight loader issues nothing, so the MMA thread's
  // stage wait runs out and the timeout path (status bit, abort of the
  // other roles, drain, TMEM release) executes.
  int selftest_stall;
};

__global__ void __launch_bounds__(kFThreads, 1)
ffn_fused_kernel(const __grid_constant__ CUtensorMap tmap_w13, const __grid_constant__ CUtensorMap tmap_wd,
                 FfnFusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = smem;                               // [D / 64][128 rows x 64]
  uint8_t* ring = smem + kFXBytes;                  // kFStages x 32 KB
  uint8_t* acts = ring + kFStages * kFStageBytes;   // 2 buffers x [2][128 rows x 64]

  __shared__ __align__(8) uint64_t full_bar[kFStages];
  __shared__ __align__(8) uint64_t empty_bar[kFStages];
  __shared__ __align__(8) uint64_t x_full, x_empty, acc1_full, acc1_empty, acc2_full, acc2_empty, drain_bar;
  __shared__ __align__(8) uint64_t act_full[2], act_free[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksub = a.D / kBK;                  // 64-column sub-tiles of x (= k-slices of the gate/up product)
  const int np = a.I / 128;                    // 128-column pieces of the intermediate
  constexpr int kEpiThreads = 32 * kFEpiWarps;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kFStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&x_full), 32 * kFGatherWarps);  // every gather lane, once its copies land
    ptx::mbar_init(ptx::smem_u32(&x_empty), 1);
    ptx::mbar_init(ptx::smem_u32(&acc1_full), 1);
    ptx::mbar_init(ptx::smem_u32(&acc1_empty), kEpiThreads);
    ptx::mbar_init(ptx::smem_u32(&acc2_full), 1);
    ptx::mbar_init(ptx::smem_u32(&acc2_empty), kEpiThreads);
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&act_full[b]), kEpiThreads);
      ptx::mbar_init(ptx::smem_u32(&act_free[b]), 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), 512);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_w13);
    ptx::prefetch_tmap(&tmap_wd);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  // tile t -> its group's rows [row0, hi): the largest g with tiles[g] <= t
  // (binary search in the prefix table), then its block within the group
  const int n_tiles = __ldg(a.tiles + a.groups);
  auto decode = [&](int t, int* row0, int* hi) {
    int lo_g = 0, hi_g = a.groups - 1;
    while (lo_g < hi_g) {
      const int mid = (lo_g + hi_g + 1) >> 1;
      if (__ldg(a.tiles + mid) <= t) lo_g = mid; else hi_g = mid - 1;
    }
    const int r0 = __ldg(a.offsets + lo_g), r1 = __ldg(a.offsets + lo_g + 1);
    *row0 = r0 + (t - __ldg(a.tiles + lo_g)) * kBM;
    *hi = r1;
    return lo_g;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_par = 0;
      bool ok = true;
      auto next_slot = [&](uint32_t bytes) -> uint32_t {
        if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, a.wait_ns)) return 0;
        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full_bar[stage]), bytes);
        filled |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        return ptx::smem_u32(ring + stage * kFStageBytes);
      };
      auto advance = [&]() {
        if (++stage == kFStages) { stage = 0; phase ^= 1; }
      };
      auto push_w13 = [&](int g, int p) {  // rows [g*2I + 256p, +256), one k-slice per stage
        for (int kb = 0; kb < ksub; ++kb) {
          const uint32_t sa = next_slot(static_cast<uint32_t>(kFStageBytes));
          if (sa == 0) return false;
          ptx::tma_load_2d(sa, &tmap_w13, kb * kBK, g * 2 * a.I + 256 * p, ptx::smem_u32(&full_bar[stage]), pol);
          advance();
        }
        return true;
      };
      auto push_wd = [&](int g, int p) {  // W_down rows [g*D, +D), columns [128p, +128), 64 per stage
        for (int s = 0; s < 2; ++s) {
          const uint32_t sa = next_slot(static_cast<uint32_t>(a.D) * 128u);
          if (sa == 0) return false;
          ptx::tma_load_2d(sa, &tmap_wd, 128 * p + 64 * s, g * a.D, ptx::smem_u32(&full_bar[stage]), pol);
          advance();
        }
        return true;
      };
      // tiles are decoded once each, the next one while this one's first
      // gate/up slices wait for ring slots (a decode is a binary search of
      // dependent global loads; done at the top of each tile it delayed the
      // tile's first loads)
      int g = 0, r0, r1;
      if (static_cast<int>(blockIdx.x) < n_tiles) g = decode(blockIdx.x, &r0, &r1);
      for (int t = blockIdx.x; t < n_tiles && ok && !a.selftest_stall; t += gridDim.x) {
        int g_n = 0;
        {
          // ring order: w13(0), w13(1), wd(0), w13(2), wd(1), ..., w13(np-1), wd(np-2), wd(np-1)
          ok = push_w13(g, 0);
          if (t + static_cast<int>(gridDim.x) < n_tiles) g_n = decode(t + gridDim.x, &r0, &r1);
          for (int p = 1; p < np && ok; ++p) ok = push_w13(g, p) && push_wd(g, p - 1);
          if (ok) ok = push_wd(g, np - 1);
        }
        g = g_n;
      }
      if (!ok) {
        atomicOr(a.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
      }
      // drain: every issued load must have landed before the CTA may exit
      const volatile int never = 0;
      for (int s = 0; s < kFStages; ++s)
        if ((filled & (1u << s)) &&
            !ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (last_par >> s) & 1u, &never, a.wait_ns))
          atomicOr(a.status, MOE_DEV_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc1 = ptx::idesc_bf16_m128(256);
      const uint32_t idesc2 = ptx::idesc_bf16_m128(a.D);
      const uint32_t t_acc1 = tmem_base, t_acc2 = tmem_base + kAcc2Col;
      int stage = 0;
      uint32_t phase = 0, tiles = 0, q1 = 0, q2 = 0;  // tiles, gate/up pieces and down pieces issued
      bool ok = true;
      auto wait = [&](uint64_t& bar, uint32_t parity) {
        if (!ok) return false;
        if (!ptx::mbar_wait(ptx::smem_u32(&bar), parity, &s_abort, a.wait_ns)) ok = false;
        ptx::tc_fence_after();
        return ok;
      };
      auto mma1 = [&](bool last) {  // gate/up piece q1 into acc1, once the epilogue has read the previous one
        if (!wait(acc1_empty, (q1 & 1) ^ 1)) return false;
        for (int kb = 0; kb < ksub; ++kb) {
          if (!wait(full_bar[stage], phase)) return false;
          const uint32_t sb = ptx::smem_u32(ring + stage * kFStageBytes);
          const uint32_t sa = ptx::smem_u32(xs + kb * kFSub);
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk)
            ptx::mma_bf16(t_acc1, ptx::sw128_desc(sa + kk * 32), ptx::sw128_desc(sb + kk * 32), idesc1,
                          (kb | kk) != 0 ? 1u : 0u);
          ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
          if (++stage == kFStages) { stage = 0; phase ^= 1; }
        }
        ptx::mma_commit(ptx::smem_u32(&acc1_full));
        if (last) ptx::mma_commit(ptx::smem_u32(&x_empty));  // the tile's last reader of x
        ++q1;
        return true;
      };
      auto mma2 = [&](bool first, bool last) {  // down piece q2 (act buffer q2 % 2) into acc2
        const int b = q2 & 1;
        if (!wait(act_full[b], (q2 >> 1) & 1)) return false;
        if (first && !wait(acc2_empty, (tiles & 1) ^ 1)) return false;
        for (int s = 0; s < 2; ++s) {
          if (!wait(full_bar[stage], phase)) return false;
          const uint32_t sa = ptx::smem_u32(acts + b * kFActBytes + s * kFSub);
          const uint32_t sb = ptx::smem_u32(ring + stage * kFStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk)
            ptx::mma_bf16(t_acc2, ptx::sw128_desc(sa + kk * 32), ptx::sw128_desc(sb + kk * 32), idesc2,
                          (first && s == 0 && kk == 0) ? 0u : 1u);
          ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
          if (++stage == kFStages) { stage = 0; phase ^= 1; }
        }
        ptx::mma_commit(ptx::smem_u32(&act_free[b]));
        if (last) ptx::mma_commit(ptx::smem_u32(&acc2_full));
        ++q2;
        return true;
      };
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        {
          if (!wait(x_full, tiles & 1)) break;
          if (!mma1(np == 1)) break;
          for (int p = 1; p < np && ok; ++p) {
            // order: gate/up(p-1), down(p-2), gate/up(p), down(p-1): the
            // epilogue reads acc1 for piece p-1 while the pipe runs down(p-2),
            // and forms act(p-1) while it runs gate/up(p)
            if (!mma1(p == np - 1)) break;
            if (!mma2(p == 1, false)) break;
          }
          if (ok) mma2(np == 1, true);
          ++tiles;
        }
      }
      if (!ok) {
        atomicOr(a.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      ptx::mma_commit(ptx::smem_u32(&drain_bar));
      const volatile int never = 0;
      if (!ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &never, a.wait_ns)) atomicOr(a.status, MOE_DEV_TIMEOUT);
    }
  } else if (warp < kFGatherWarp) {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int part = (warp - 2) / 4;  // 0: chunk 2p, first half of y; 1: chunk 2p+1, second half
    const int r = quad * 32 + lane;   // tile row = TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const int yh = a.D / 2;           // y columns per part (a multiple of 32)
    uint32_t tiles = 0, q = 0;
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
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tiles) {
      int row0, hi;
      decode(t, &row0, &hi);
      {
        for (int p = 0; p < np && ok; ++p, ++q) {
          if (!wait(acc1_full, q & 1)) break;
          // this part's chunk: gate columns [128 part, +64), up columns [128 part + 64, +64)
          uint32_t pk[32];
          {
            uint32_t gr[64], ur[64];
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              ptx::tmem_ld16(lane_addr + part * 128 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(gr + 16 * c));
              ptx::tmem_ld16(lane_addr + part * 128 + 64 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(ur + 16 * c));
            }
            ptx::tmem_ld_wait();  // one wait for all eight loads: acc1 is held for the loads alone
            // acc1 may take the next piece's products while this warp finishes
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&acc1_empty));
#pragma unroll
            for (int i = 0; i < 32; ++i)
              pk[i] = pack_bf16x2(silu(__uint_as_float(gr[2 * i])) * __uint_as_float(ur[2 * i]),
                                  silu(__uint_as_float(gr[2 * i + 1])) * __uint_as_float(ur[2 * i + 1]));
          }
          const int b = q & 1;
          if (!wait(act_free[b], ((q >> 1) & 1) ^ 1)) break;
          const uint32_t dst = ptx::smem_u32(acts + b * kFActBytes + part * kFSub) + static_cast<uint32_t>(r) * 128u;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            ptx::st_shared_v4(dst + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(r) & 7u)) << 4),
                              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
          ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core (async proxy) reads
          ptx::mbar_arrive(ptx::smem_u32(&act_full[b]));
        }
        if (!ok) break;
        // this part's half of the tile's y rows: acc2 -> bf16, the accumulator handed back, then stored
        if (!wait(acc2_full, tiles & 1)) break;
        uint32_t yk[kFMaxD / 4];
#pragma unroll
        for (int col = 0; col < kFMaxD / 2; col += 32) {
          if (col < yh) {
            float v[32];
            __syncwarp();
            tmem_ld32(lane_addr + kAcc2Col + part * yh + col, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) yk[col / 2 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&acc2_empty));
        const int row = row0 + r;
        if (row < hi) {
          uint4* dst = reinterpret_cast<uint4*>(a.y + static_cast<int64_t>(row) * a.D + part * yh);
#pragma unroll
          for (int c = 0; c < kFMaxD / 16; ++c)
            if (c < yh / 8) dst[c] = make_uint4(yk[4 * c], yk[4 * c + 1], yk[4 * c + 2], yk[4 * c + 3]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- gather
    // Each tile's x rows, head slice of x by source token, straight into the
    // 128-byte-swizzled sub-tiles the MMA descriptors expect: 8 lanes per
    // 128-byte row slice, 4 rows per warp instruction.  Each lane waits for
    // its own copies, fences the generic proxy against the tensor core's
    // async-proxy reads and arrives on x_full (a fence in the MMA thread
    // instead would sit on the tensor pipe's critical path at every tile).
    // x is read from L2 (each token's head slice is read by its top-k
    // experts), x_perm never exists.
    const uint64_t pol = ptx::policy_evict_last();
    const int chunk = lane & 7, rsub = lane >> 3;
    const int rbase = (warp - kFGatherWarp) * kFGatherRows;  // this warp's first tile row
    uint32_t tiles = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tiles) {
      int row0, hi;
      const int g = decode(t, &row0, &hi);
      const int64_t col0 = static_cast<int64_t>(g / a.head_groups) * a.D + chunk * 8;
      // this warp's source tokens, one per lane per 32 rows in one coalesced
      // pass (-1: past the group's rows, or out of range and flagged)
      int toks[kFGatherRows / 32];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < kFGatherRows / 32; ++i) {
        const int row = row0 + rbase + 32 * i + lane;
        int tok = row < hi ? __ldg(a.src + row) : -1;
        if (row < hi && (tok < 0 || tok >= a.T)) {
          bad = true;
          tok = -1;
        }
        toks[i] = tok;
      }
      if (bad) atomicOr(a.status, MOE_DEV_BAD_SOURCE_ROW);
      // (the decode and the token loads above do not need x free); the
      // previous tile's gate/up products are done with the x sub-tiles
      const bool got = ptx::mbar_wait(ptx::smem_u32(&x_empty), (tiles & 1) ^ 1, &s_abort, a.wait_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicOr(a.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
        ok = false;
        break;
      }
#pragma unroll
      for (int j = 0; j < kFGatherRows / 4; ++j) {
        const int r = rbase + 4 * j + rsub;  // r - rbase = 32 * (j / 8) + (4 * (j % 8) + rsub)
        const int tok = __shfl_sync(0xffffffffu, toks[j / 8], 4 * (j % 8) + rsub);
        const bool v = tok >= 0;
        const uint16_t* src = a.x + static_cast<int64_t>(v ? tok : 0) * a.x_ld + col0;
        const uint32_t dst = ptx::smem_u32(xs) + static_cast<uint32_t>(r) * 128u +
                             ((static_cast<uint32_t>(chunk) ^ (static_cast<uint32_t>(r) & 7u)) << 4);
        for (int kb = 0; kb < ksub; ++kb)
          ptx::cp_async_16(dst + static_cast<uint32_t>(kb * kFSub), src + kb * kBK, v ? 16u : 0u, pol);
      }
      // this lane's copies land, are ordered before the tensor core's
      // (async-proxy) reads by this lane's own proxy fence, then x_full
      ptx::cp_async_wait_all();
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_u32(&x_full));
    }
    ptx::cp_async_wait_all();  // (an early exit leaves no copy in flight)
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

// tiles[g] = exclusive prefix over the groups of their 128-row tile counts,
// tiles[groups] = the total.  A group with bad offsets (negative, decreasing
// or past `rows`) counts no tiles and sets MOE_DEV_BAD_OFFSETS.  One block.
__global__ void __launch_bounds__(1024) tile_prefix_kernel(const int* __restrict__ offsets, int groups, int rows,
                                                            int* __restrict__ tiles, int* status) {
  __shared__ int warp_sum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (groups + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
  const int g0 = min(static_cast<int>(threadIdx.x) * per, groups), g1 = min(g0 + per, groups);
  auto count = [&](int g, bool* bad) {
    const int r0 = __ldg(offsets + g), r1 = __ldg(offsets + g + 1);
    if (r0 < 0 || r1 < r0 || r1 > rows) {
      *bad = true;
      return 0;
    }
    return (r1 - r0 + kBM - 1) / kBM;
  };
  bool bad = false;
  int sum = 0;
  for (int g = g0; g < g1; ++g) sum += count(g, &bad);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int n = static_cast<int>(blockDim.x) >> 5;
    const int v = lane < n ? warp_sum[lane] : 0;
    int w = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < n) warp_sum[lane] = w - v;  // exclusive prefix of the warps' sums
  }
  __syncthreads();
  int run = warp_sum[warp] + incl - sum;
  for (int g = g0; g < g1; ++g) {
    tiles[g] = run;
    run += count(g, &bad);
  }
  if (threadIdx.x == blockDim.x - 1) tiles[groups] = run;  // the last range ends at `groups`: run = total
  if (bad) atomicOr(status, MOE_DEV_BAD_OFFSETS);
}

}  // namespace

bool ffn_fused_supported(int D, int I) { return D % 64 == 0 && D >= 64 && D <= kFMaxD && I % 128 == 0 && I >= 128; }

namespace {

int run_ffn_fused(const CUtensorMap& tw, const CUtensorMap& td, const FfnFusedArgs& fa, int grid,
                  cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  if (!smem_attr_ready(ffn_fused_kernel, kFDynBytes, smem_set)) return MOE_ERR_CUDA;
  // at most one CTA per SM; a CTA with no tile returns at once
  ffn_fused_kernel<<<grid, kFThreads, kFDynBytes, stream>>>(tw, td, fa);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int launch_ffn_fused(const FfnArgs& a, cudaStream_t stream) {
  if (!ffn_fused_supported(a.d, a.I)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.rows >= (int64_t{1} << 31) || a.T >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.x == nullptr || a.src_token == nullptr || a.head_groups < 1 || a.x_ld < a.d || a.x_ld % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  CUtensorMap tw, td;
  // w13: 256 rows (two 64-column chunks' gate | up) per load; W_down: D rows per load
  if (!make_tmap_bf16_2d(&tw, a.w13, a.d, static_cast<uint64_t>(a.E) * 2 * a.I, kBK, 256)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, a.w_down, a.I, static_cast<uint64_t>(a.E) * a.d, kBK, a.d)) return MOE_ERR_CUDA;
  if (a.tiles == nullptr || a.E < 1) return MOE_ERR_INVALID_ARG;
  tile_prefix_kernel<<<1, 1024, 0, stream>>>(a.offsets, a.E, static_cast<int>(a.rows), a.tiles, a.status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  FfnFusedArgs fa{};
  fa.offsets = a.offsets;
  fa.tiles = a.tiles;
  fa.groups = a.E;
  fa.rows = static_cast<int>(a.rows);
  fa.x = a.x;
  fa.x_ld = a.x_ld;
  fa.src = a.src_token;
  fa.T = static_cast<int>(a.T);
  fa.head_groups = a.head_groups;
  fa.D = a.d;
  fa.I = a.I;
  fa.y = a.y_perm;
  fa.status = a.status;
  fa.wait_ns = kWaitLimitNs;
  return run_ffn_fused(tw, td, fa, a.sm_count, stream);
}

// The fused kernel on one 128-row tile (D = 64, I = 128, all rows reading
// token 0) with its weight loader stalled; `scratch` holds the tile's
// buffers (96 KB, 16-byte aligned).
int launch_ffn_fused_selftest(uint8_t* scratch, int* status, uint64_t limit_ns, cudaStream_t stream) {
  constexpr int D = 64, I = 128, R = 128;
  uint16_t* x = reinterpret_cast<uint16_t*>(scratch);              // [R, D]
  uint16_t* w13 = x + R * D;                                       // [2I, D]
  uint16_t* wd = w13 + 2 * I * D;                                  // [D, I]
  uint16_t* y = wd + D * I;                                        // [R, D]
  int* src = reinterpret_cast<int*>(y + R * D);                    // [R]
  int* offsets = src + R;                                          // [2]
  int* tiles = offsets + 4;                                        // [2]
  static const int kOffsets[2] = {0, R};
  if (cudaMemsetAsync(scratch, 0, reinterpret_cast<uint8_t*>(offsets) - scratch, stream) != cudaSuccess ||
      cudaMemcpyAsync(offsets, kOffsets, sizeof(kOffsets), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  CUtensorMap tw, td;
  if (!make_tmap_bf16_2d(&tw, w13, D, 2 * I, kBK, 256)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, wd, I, D, kBK, D)) return MOE_ERR_CUDA;
  tile_prefix_kernel<<<1, 1024, 0, stream>>>(offsets, 1, R, tiles, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  FfnFusedArgs fa{};
  fa.offsets = offsets;
  fa.tiles = tiles;
  fa.groups = 1;
  fa.rows = R;
  fa.x = x;
  fa.x_ld = D;
  fa.src = src;
  fa.T = R;
  fa.head_groups = 1;
  fa.D = D;
  fa.I = I;
  fa.y = y;
  fa.status = status;
  fa.wait_ns = limit_ns;
  fa.selftest_stall = 1;
  return run_ffn_fused(tw, td, fa, 1, stream);
}

}  // namespace moe
