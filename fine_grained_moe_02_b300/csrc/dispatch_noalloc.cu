// moe_dispatch_noalloc: the sorting stage (histogram, scan, rank assignment,
// row gather) for callers that cannot allocate device memory.  Its scratch is
// a fixed array in the library's own device image instead of a caller
// workspace; see include/moe.h for the contract.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "moe.h"

namespace {

// Per-block expert counters, ceil(T / 2048) * E cells.
constexpr int64_t kNoAllocMaxCells = 65536;
constexpr int64_t kSinkInts = 64;  // status sink when the caller passes no status word

// Lives for as long as the library is loaded, on every GPU that loads it.
static __device__ __align__(256) int32_t g_dispatch_scratch[kSinkInts + kNoAllocMaxCells];

// Device address of g_dispatch_scratch in the current context.  Host code may
// not use the symbol itself (on the host it names a stand-in, not device
// memory).  The address is looked up on every call rather than cached per
// device: a cudaDeviceReset, or another context on the same device, loads
// the module again at a different address, and a cached pointer would then
// aim at memory that is no longer this array.  The lookup allocates nothing;
// the first one in a context loads the module there.
int scratch_address(int32_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
  *out = static_cast<int32_t*>(p);
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_dispatch_noalloc(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx,
                                    int32_t* offsets, int32_t* row_of, int32_t* src_token, moe_bf16* x_perm,
                                    int32_t* status, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || topk_idx == nullptr || offsets == nullptr || row_of == nullptr || src_token == nullptr ||
      x_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(offsets) || !aligned16(row_of) ||
      !aligned16(src_token) || !aligned16(x_perm) || (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u)))
    return MOE_ERR_MISALIGNED;
  // the counters need ceil(T / 2048) * E cells
  const int64_t cells = static_cast<int64_t>(moe::dispatch_counter_cells(dims->T, dims->E));
  if (cells > kNoAllocMaxCells) return MOE_ERR_UNSUPPORTED_SHAPE;

  int32_t* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != MOE_OK) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return MOE_ERR_CUDA;

  // Every cell the kernels read is written earlier in the same call (the
  // histogram pass writes all counters before the assign pass reads them),
  // so nothing is cleared; the sink word is written but never read.
  moe::DispatchArgs a{};
  a.x = x;
  a.topk_idx = topk_idx;
  a.T = dims->T;
  a.d = dims->d;
  a.k = dims->top_k;
  a.E = dims->E;
  a.offsets = offsets;
  a.row_of = row_of;
  a.src_token = src_token;
  a.x_perm = x_perm;
  a.block_counts = scratch + kSinkInts;
  a.status = status != nullptr ? status : scratch;
  a.sm_count = sms;
  return moe::launch_dispatch(a, static_cast<cudaStream_t>(stream));
}
