// Persistent tcgen05 GEMM engine for sm_103a: D = A * B^T over ragged row
// groups, bf16 operands, fp32 accumulation in tensor memory.
//
//   A: rows of a [M_total, K] bf16 matrix, loaded by TMA (128-byte swizzle)
//   B: rows of a [groups * N, K_B] bf16 matrix (group g uses rows g*N ..),
//      the k coordinate of B is k mod K_B (lets one B serve a K = c*K_B sweep)
//   groups: device offsets[G + 1]; group g owns A rows [offsets[g], offsets[g+1])
//
// One CTA per SM, 64 + 32 * Epi::kWarps (+ 32 * GW) threads:
//   warp 0       TMA producer (one lane): fills a STAGES-deep shared-memory ring
//   warp 1       MMA issuer (one lane) and TMEM owner: tcgen05.mma 128 x BN x 16
//   warps 2..    epilogue (4 or 8 warps: warp w reads TMEM lane quadrant w % 4):
//                tcgen05.ld the accumulator, apply Epi, store to HBM
//   last GW      A gather warps (GW > 0): cp.async row copies instead of TMA
// The accumulator is double-buffered in TMEM so the epilogue of tile i
// overlaps the main loop of tile i+1.  Tiles are handed out statically
// (tile = blockIdx.x + i * gridDim.x) in group-major, m-major, n-minor order
// so that CTAs running at the same time share A and B tiles through L2.
//
// Every wait is bounded (see ptx::mbar_wait): on a timeout the kernel sets
// MOE_DEV_TIMEOUT in the status word, the other roles stop, in-flight TMA
// loads and MMAs are drained (again with a limit), TMEM is freed and the
// kernel returns.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "internal.h"
#include "moe.h"
#include "ptx.cuh"

namespace moe {

constexpr int kBM = 128;          // tile rows (UMMA M)
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row of bf16
constexpr int kUK = 16;           // k per tcgen05.mma (kind::f16)
constexpr int kMaxGroups = kMaxGemmGroups;  // tile prefix table in shared memory
constexpr int kGemmThreads = 192;  // producer + MMA warps and four epilogue warps

// Threads of a GEMM CTA: producer and MMA warps, Epi::kWarps epilogue warps
// (4, or 8 when two warps share each TMEM lane quadrant) and GW gather warps.
template <class Epi, int GW>
constexpr int gemm_threads() {
  return 64 + 32 * Epi::kWarps + 32 * GW;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kOutChunkBytes = 32 * 128;          // 32 rows x 64 bf16

struct GemmShape {
  int K;            // reduction length (A's columns)
  int K_B;          // B's columns; B's k coordinate is k % K_B
  int N;            // output columns per group (multiple of BN)
  int groups;       // number of row groups (1 for a dense GEMM)
  const int* offsets;  // device [groups + 1], or nullptr: one group of rows [0, M)
  int M;            // rows when offsets == nullptr; row capacity of A otherwise
  int* status;      // device status word
  // Row gather for A (kernels with gather warps, GW > 0): logical A row r is
  // row a_gather[r] of a_src, a row-major [*, K] bf16 matrix with a_ld
  // elements per row; tmap_a is not used.
  const int* a_gather;
  // A's k coordinate is k % K_A (0 means K): one A tile serves a K = c*K_A
  // sweep (the folded router reads x twice, against W_eff's hi and lo halves).
  int K_A;
  // Limit of every pipeline wait (0: kWaitLimitNs).
  uint64_t wait_limit_ns;
  // Self-test only: the producer issues no loads, so the other roles' waits
  // run out and the timeout path (status bit, drain, TMEM release) executes.
  int selftest_stall;
  // Batched dense mode (offsets == nullptr, batched != 0): `groups`
  // independent problems over the same M rows of A; problem g reads A's
  // columns from g * a_col_stride and B's rows from g * b_group_rows.
  int batched;
  int a_col_stride;
  int b_group_rows;
  const uint16_t* a_src;
  int64_t a_ld;
  int a_src_rows;   // rows of a_src: a gathered index outside [0, a_src_rows) reads zeros
};

// Gather warps: the A operand's rows are fetched by 32*GW threads with 16-byte
// cp.async copies, 8 lanes per 128-byte row slice (4 whole rows per warp
// instruction); each thread hands the stage's full barrier an arrival that
// fires when its copies have landed (cp.async.mbarrier.arrive.noinc) and goes
// on to the next stage at once.  The MMA thread, having seen the barrier
// complete, orders those generic-proxy writes before the tensor core's
// async-proxy reads with a proxy fence of its own.

template <int BN>
struct GemmSmem {
  static constexpr int kStages = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
  static constexpr int kAccStride = kTmemCols / 2;  // column offset of accumulator buffer 1
  // one 32-row x 64-column bf16 staging chunk (4 KB, 128-byte swizzled) per epilogue warp
  static constexpr int kOutBytes = 4 * kOutChunkBytes;
  // ring + output staging + 1 KB slack for the manual 1024-byte alignment
  static constexpr int kDynBytes = kStages * kStageBytes + kOutBytes + 1024;
};

// What an epilogue needs besides the accumulator: the output tensor map, this
// warp's staging buffer and whether a bulk store from it may still be reading.
struct EpiCtx {
  const CUtensorMap* tmap;
  uint32_t stage;   // shared address of this warp's 4 KB staging chunk
  int lane;
  int quad;         // TMEM lane quadrant = rows [32*quad, 32*quad + 32) of the tile
  bool pending;     // lane 0 has a committed bulk store that may still read `stage`
  uint32_t tempty;  // shared address of the current accumulator's "empty" barrier
  bool released;    // this warp has already arrived on `tempty` for the current tile
  int part;         // with 8 epilogue warps: which of the quadrant's two warps (0, 1)
  uint32_t scratch; // shared address of the epilogue scratch (the staging area)
  // hand-off between a quadrant's two warps (8 epilogue warps): "filled" and
  // "free" mbarriers of the quadrant (32 arrivals each), uses so far, and the
  // bounds of every wait; `failed` reports a wait that ran out
  uint32_t hand_full, hand_free;
  uint32_t hand_uses;
  const volatile int* abort;
  uint64_t wait_ns;
  bool failed;
  // cycles a store-heavy epilogue waits between handing the accumulator back
  // and its first store (0 on the CTA's last tile): a quarter to 0.7 of the
  // next tile's MMA time, by lane quadrant, so the tile's stores are spread
  // over the next tile's operand loads rather than meeting their start
  uint32_t store_delay;
};

struct TileCoord {
  int group, m_blk, n_blk;
  int row0;      // first A row of the tile
  int row_end;   // end of the group's rows (exclusive)
};

// First A row of group g (g = groups: the end of the last group): the device
// offsets, or the dense layouts (one group of M rows; batched: g * M).
struct GroupRows {
  const int* offsets;
  int batched;
  int M;
  __device__ __forceinline__ int operator()(int g) const {
    return offsets ? __ldg(offsets + g) : (batched ? g * M : (g == 0 ? 0 : M));
  }
};

template <int BN>
__device__ __forceinline__ TileCoord decode_tile(int tile, const GroupRows& rows, const int* s_tile, int groups,
                                                 int n_tiles) {
  // largest g with s_tile[g] <= tile
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tile[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  TileCoord c;
  c.group = lo;
  const int local = tile - s_tile[lo];
  c.m_blk = local / n_tiles;
  c.n_blk = local - c.m_blk * n_tiles;
  c.row0 = rows(lo) + c.m_blk * kBM;
  c.row_end = rows(lo + 1);
  return c;
}

// Epi must provide:
//   struct Params;
//   template <int BN> static __device__ void run(const Params&, const TileCoord&, uint32_t taddr,
//                                                 int row_in_tile, EpiCtx&);
// taddr addresses this thread's lane (= tile row) at the accumulator's column 0.
template <int BN, class Epi, int GW = 0>
__global__ void __launch_bounds__(gemm_threads<Epi, GW>(), 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
               const __grid_constant__ CUtensorMap tmap_d, GemmShape shape, typename Epi::Params ep) {
  using S = GemmSmem<BN>;
  constexpr int STAGES = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t hand_bar[8];  // 8 epilogue warps: per quadrant "filled" (0-3) and "free" (4-7)
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_tile[kMaxGroups + 1];
  __shared__ int s_total;
  __shared__ int s_bad;

  static_assert(kBM % (4 * (GW > 0 ? GW : 1)) == 0, "gather warps cover the tile's rows evenly");
  static_assert(GW % 2 == 0, "a gather thread's rows r, r + 4*GW, ... share one 128-byte swizzle phase");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = shape.N / BN;
  const int groups = shape.groups;
  const int first_tile = static_cast<int>(blockIdx.x);
  const int tile_step = static_cast<int>(gridDim.x);

  // ---- group table: tile counts of the groups (all threads; group rows come
  // from the offsets in global memory, and again when a tile is decoded),
  // then their exclusive prefix (warp 0, each lane summing a contiguous run)
  // (batched dense mode: every group spans rows [0, M); decode_tile maps them)
  const GroupRows rows{shape.offsets, shape.batched, shape.M};
  const int row_limit = shape.batched ? groups * shape.M : shape.M;
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_bad = 0;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < groups; g += blockDim.x) {
    const int a = rows(g), b = rows(g + 1);
    int cnt = 0;
    if (a < 0 || b < a || b > row_limit) s_bad = 1;
    else cnt = ((b - a + kBM - 1) / kBM) * n_tiles;
    s_tile[g] = cnt;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (groups + 31) / 32;
    const int g0 = min(lane * per, groups), g1 = min(g0 + per, groups);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += s_tile[g];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int g = g0; g < g1; ++g) {
      const int c = s_tile[g];
      s_tile[g] = run;
      run += c;
    }
    if (lane == 31) {
      s_tile[groups] = incl;
      s_total = s_bad ? 0 : incl;
      if (s_bad && blockIdx.x == 0) atomicOr(shape.status, MOE_DEV_BAD_OFFSETS);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1 + 32 * GW);  // the B (+A) loader, every gather thread
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), 32 * Epi::kWarps);
    }
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    for (int q = 0; q < 8; ++q) ptx::mbar_init(ptx::smem_u32(&hand_bar[q]), 32);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), S::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
    ptx::prefetch_tmap(&tmap_d);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const uint32_t tmem_base = s_tmem;
  const int total = s_total;
  const int num_kb = shape.K / kBK;
  const uint64_t wait_ns = shape.wait_limit_ns ? shape.wait_limit_ns : kWaitLimitNs;

  constexpr int kEpiEnd = 2 + Epi::kWarps;  // first warp after the epilogue warps
  static_assert(Epi::kWarps == 4 || Epi::kWarps == 8, "one or two epilogue warps per TMEM lane quadrant");
  if (GW > 0 && warp >= kEpiEnd) {
    // -------------------------------------------------------- A gather warps
    const int gt = static_cast<int>(threadIdx.x) - 32 * kEpiEnd;  // 0 .. 32*GW - 1
    constexpr int kRowStep = 4 * (GW > 0 ? GW : 1);               // rows per instruction of all gather warps
    constexpr int kRowsPer = kBM / kRowStep;                      // rows per thread per k-slice
    const int chunk = gt & 7;                                     // this lane's 16-byte chunk of a row slice
    const int r_first = gt >> 3;                                  // rows r_first + j * kRowStep
    const uint32_t dst_off = static_cast<uint32_t>(r_first) * 128u +
                             ((static_cast<uint32_t>(chunk) ^ (static_cast<uint32_t>(r_first) & 7u)) << 4);
    const uint64_t pol = ptx::policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = first_tile; tile < total && ok; tile += tile_step) {
      const TileCoord c = decode_tile<BN>(tile, rows, s_tile, groups, n_tiles);
      const uint16_t* src[kRowsPer];
      uint32_t valid = 0;
      bool bad_row = false;
#pragma unroll
      for (int j = 0; j < kRowsPer; ++j) {
        const int row = c.row0 + r_first + j * kRowStep;
        int tok = row < c.row_end ? __ldg(shape.a_gather + row) : -1;
        if (row < c.row_end && (tok < 0 || tok >= shape.a_src_rows)) bad_row = true;
        const bool v = tok >= 0 && tok < shape.a_src_rows;
        if (!v) tok = 0;
        src[j] = shape.a_src + static_cast<int64_t>(tok) * shape.a_ld + chunk * 8;
        valid |= (v ? 1u : 0u) << j;
      }
      if (bad_row) atomicOr(shape.status, MOE_DEV_BAD_SOURCE_ROW);
      for (int kb = 0; kb < num_kb; ++kb) {
        bool got = true;
        if (lane == 0) got = ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, wait_ns);
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        const uint32_t sa = ptx::smem_u32(smem + stage * S::kStageBytes) + dst_off;
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j)  // row r_first + j*kRowStep keeps the swizzle of r_first (kRowStep % 8 == 0)
          ptx::cp_async_16(sa + static_cast<uint32_t>(j * kRowStep) * 128u, src[j] + kb * kBK,
                           ((valid >> j) & 1u) ? 16u : 0u, pol);
        ptx::cp_async_mbar_arrive_noinc(ptx::smem_u32(&full_bar[stage]));
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok && lane == 0) {
      atomicOr(shape.status, MOE_DEV_TIMEOUT);
      s_abort = 1;
    }
    // drain: this thread's copies land before it may exit (their barrier
    // arrivals are awaited by the producer's drain)
    ptx::cp_async_wait_all();
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      // Both operands evict_last: an A tile is read by the n_tiles CTAs that
      // share its rows at slightly different times and must survive until the
      // last one (with evict_normal on A, expert GEMM-1 on the clip workload
      // re-read 22% of x_perm from DRAM); B is reused by every m-block of the group.
      const uint64_t pol_a = ptx::policy_evict_last();
      const uint64_t pol_b = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;       // bit s: stage s was filled at least once
      uint32_t last_par = 0;     // bit s: parity of the last fill of stage s
      bool ok = true;
      for (int tile = first_tile; tile < total && ok && !shape.selftest_stall; tile += tile_step) {
        const TileCoord c = decode_tile<BN>(tile, rows, s_tile, groups, n_tiles);
        const int b_row = c.group * (shape.b_group_rows ? shape.b_group_rows : shape.N) + c.n_blk * BN;
        const int a_row = shape.batched ? c.row0 - c.group * shape.M : c.row0;
        const int a_col = shape.batched ? c.group * shape.a_col_stride : 0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
          ptx::mbar_arrive_expect_tx(fb, GW > 0 ? S::kBBytes : S::kStageBytes);  // gathered A arrives by cp.async
          const uint32_t sa = ptx::smem_u32(smem + stage * S::kStageBytes);
          const uint32_t sb = sa + S::kABytes;
          const int k = kb * kBK;
          if (GW == 0)
            ptx::tma_load_2d(sa, &tmap_a, a_col + (shape.K_A > 0 ? k % shape.K_A : k), a_row, fb, pol_a);
          ptx::tma_load_2d(sb, &tmap_b, k % shape.K_B, b_row, fb, pol_b);
          filled |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        atomicOr(shape.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
      }
      // drain: every issued load must have landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s) {
        if (filled & (1u << s)) {
          const volatile int never = 0;
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (last_par >> s) & 1u, &never, wait_ns))
            atomicOr(shape.status, MOE_DEV_TIMEOUT);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_m128(BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = first_tile; tile < total && ok; tile += tile_step) {
        if (!ptx::mbar_wait(ptx::smem_u32(&tempty_bar[acc]), acc_phase ^ 1, &s_abort, wait_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * S::kAccStride);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), phase, &s_abort, wait_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          if (GW > 0) ptx::fence_proxy_async_smem();  // the gathered A rows were written by cp.async
          const uint32_t sa = ptx::smem_u32(smem + stage * S::kStageBytes);
          const uint32_t sb = sa + S::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk) {
            const uint64_t da = ptx::sw128_desc(sa + kk * kUK * 2);
            const uint64_t db = ptx::sw128_desc(sb + kk * kUK * 2);
            ptx::mma_bf16(d_tmem, da, db, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&tfull_bar[acc]));
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if (!ok) {
        atomicOr(shape.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      ptx::mma_commit(ptx::smem_u32(&drain_bar));
      const volatile int never = 0;
      if (!ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &never, wait_ns))
        atomicOr(shape.status, MOE_DEV_TIMEOUT);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    EpiCtx ctx{&tmap_d, ptx::smem_u32(smem + STAGES * S::kStageBytes + quad * kOutChunkBytes), lane, quad, false,
               0u, false, (warp - 2) / 4, ptx::smem_u32(smem + STAGES * S::kStageBytes),
               ptx::smem_u32(&hand_bar[quad]), ptx::smem_u32(&hand_bar[4 + quad]), 0u, &s_abort, wait_ns, false, 0u};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = first_tile; tile < total; tile += tile_step) {
      const bool ok = ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), acc_phase, &s_abort, wait_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(shape.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
        break;
      }
      ptx::tc_fence_after();
      const TileCoord c = decode_tile<BN>(tile, rows, s_tile, groups, n_tiles);
      ctx.tempty = ptx::smem_u32(&tempty_bar[acc]);
      ctx.released = false;
      // a k-slice of 128 x BN x 64 MMAs takes 2*BN cycles at the pipe's rate,
      // so num_kb * BN is half the tile's MMA time; the four lane quadrants
      // start their stores at 0.25, 0.4, 0.55 and 0.7 of it
      ctx.store_delay = tile + tile_step < total ? static_cast<uint32_t>(num_kb * BN * (5 + 3 * quad) / 10) : 0u;
      // an epilogue may hand the accumulator back itself (release_accumulator)
      // as soon as it holds the tile in registers, before its stores
      Epi::template run<BN>(ep, c, lane_addr + static_cast<uint32_t>(acc * S::kAccStride), row_in_tile, ctx);
      if (__any_sync(0xffffffffu, ctx.failed)) {
        if (lane == 0) atomicOr(shape.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
        break;
      }
      if (!ctx.released) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(ctx.tempty);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    // bulk stores read shared memory and write global memory asynchronously:
    // both must be done before the CTA exits
    if (lane == 0 && ctx.pending) ptx::bulk_wait_all();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

}  // namespace moe
