// C-ABI entry points of libmoe (declared in include/moe.h): argument checks,
// workspace layout and the order of the stages on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "moe.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// Scratch layout (offsets from ws):
//   [0, 1024)                  status word (int32 at 0)
//   dispatch counters          nblk * E int32
//   hl                         T * 2L bf16 (router latent hi | lo)
struct ScratchLayout {
  size_t disp, hl, end;
};

ScratchLayout scratch_layout(const moe_dims* d) {
  ScratchLayout s;
  const size_t L = static_cast<size_t>(d->n_heads) * d->head_dim;
  s.disp = kAlign;
  s.hl = align_up(s.disp + dispatch_scratch_bytes(d->T, d->E), kAlign);
  s.end = align_up(s.hl + static_cast<size_t>(d->T) * 2 * L * 2, kAlign);
  return s;
}

// Forward layout: scratch, then the layer's intermediates.  y_perm aliases
// x_perm (x_perm is dead once expert GEMM-1 has run).
struct ForwardLayout {
  ScratchLayout s;
  size_t idx, gate, offsets, row_of, src, xperm, act, end;
};

ForwardLayout forward_layout(const moe_dims* d) {
  ForwardLayout f;
  f.s = scratch_layout(d);
  const size_t Tk = static_cast<size_t>(d->T) * d->top_k;
  f.idx = f.s.end;
  f.gate = align_up(f.idx + Tk * 4, kAlign);
  f.offsets = align_up(f.gate + Tk * 4, kAlign);
  f.row_of = align_up(f.offsets + (static_cast<size_t>(d->E) + 1) * 4, kAlign);
  f.src = align_up(f.row_of + Tk * 4, kAlign);
  f.xperm = align_up(f.src + Tk * 4, kAlign);
  f.act = align_up(f.xperm + Tk * d->d * 2, kAlign);
  f.end = align_up(f.act + Tk * d->inter * 2, kAlign);
  return f;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int* status_ptr(void* ws) { return static_cast<int*>(ws); }

// Router choice of moe_route: small batches on chip (h stays in tensor
// memory), the rest through the two-stage path.  With few 128-token tiles the
// two-stage router's score GEMM has too few tiles to stream the latent back
// at full bandwidth.  Measured on B300 (d = 4096, E = 128, 12 x 256 heads):
// on chip 0.098 against 0.126 ms at 32 token tiles x 12 heads (T = 4096),
// slower from 40 tiles (T = 5120); the bound is 3 waves of 148 SMs.
constexpr int64_t kOnChipRouterItems = 3 * 148;

bool route_on_chip(const moe_dims* d) {
  return route_fused_supported(d->head_dim) && ((d->T + 127) / 128) * static_cast<int64_t>(d->n_heads) <= kOnChipRouterItems;
}

// moe_forward_host runs the layer over token chunks of ceil(T / n) tokens,
// n = min(ceil(T / 8192), 8).  x comes in on one stream and out goes back on
// another, so while chunk i computes on the caller's stream the copy engines
// bring chunk i+1 in and take chunk i-1 out.  With n >= 3 the first and the
// last chunk are each cut 1:3, the short piece at the end of the batch, so
// the copy in before the first compute and the compute and copy out after the
// last copy in are short.  Routing, each expert row and the combine are per
// token, so every token gets the same bits as in a single moe_forward over
// the whole batch.
constexpr int kHostChunksMax = 8;
constexpr int kHostPiecesMax = kHostChunksMax + 2;
constexpr int64_t kHostChunkMinTokens = 8192;
constexpr int kMaxDevices = 64;

int host_chunks(int64_t T) {
  return static_cast<int>(std::min<int64_t>(std::max<int64_t>((T + kHostChunkMinTokens - 1) / kHostChunkMinTokens, 1),
                                            kHostChunksMax));
}

int64_t host_chunk_tokens(int64_t T) {
  const int64_t n = host_chunks(T);
  return (T + n - 1) / n;
}

// A batch that moe_forward would route on chip runs as one piece (on-chip
// routing of a smaller piece could sum the head scores in another order);
// otherwise every piece takes the two-stage router, which gives each token
// the bits it gets in the whole batch.
bool host_one_piece(const moe_dims* d) { return route_on_chip(d); }

// The pieces the layer runs over, in token order; returns their count.
int host_pieces(int64_t T, int64_t* start, int64_t* len, bool one_piece) {
  if (one_piece) {
    start[0] = 0;
    len[0] = T;
    return 1;
  }
  const int n = host_chunks(T);
  const int64_t tc = host_chunk_tokens(T);
  int m = 0;
  int64_t t0 = 0;
  for (int i = 0; i < n && t0 < T; ++i) {
    const int64_t ti = std::min(tc, T - t0);
    if (n >= 3 && (i == 0 || i == n - 1) && ti >= 4) {
      const int64_t a = (i == 0) ? ti / 4 : ti - ti / 4;
      start[m] = t0;
      len[m++] = a;
      start[m] = t0 + a;
      len[m++] = ti - a;
    } else {
      start[m] = t0;
      len[m++] = ti;
    }
    t0 += ti;
  }
  return m;
}

// Copy streams and events of one device, created on first use and kept for
// the life of the process.  `mu` serialises moe_forward_host calls on the
// device (each call ends with all three streams drained).
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, out_end = nullptr;
  cudaEvent_t in_done[kHostPiecesMax] = {}, fwd_done[kHostPiecesMax] = {};
};

HostPipe g_host_pipe[kMaxDevices];

void host_pipe_release(HostPipe& p) {
  if (p.in) cudaStreamDestroy(p.in);
  if (p.out) cudaStreamDestroy(p.out);
  if (p.start) cudaEventDestroy(p.start);
  if (p.out_end) cudaEventDestroy(p.out_end);
  for (int i = 0; i < kHostPiecesMax; ++i) {
    if (p.in_done[i]) cudaEventDestroy(p.in_done[i]);
    if (p.fwd_done[i]) cudaEventDestroy(p.fwd_done[i]);
    p.in_done[i] = p.fwd_done[i] = nullptr;
  }
  p.in = p.out = nullptr;
  p.start = p.out_end = nullptr;
}

// Caller holds p.mu.
bool host_pipe_ready(HostPipe& p) {
  if (p.ready) return true;
  auto ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess && ev(&p.start) &&
            ev(&p.out_end);
  for (int i = 0; ok && i < kHostPiecesMax; ++i) ok = ev(&p.in_done[i]) && ev(&p.fwd_done[i]);
  if (!ok) {
    host_pipe_release(p);
    return false;
  }
  p.ready = true;
  return true;
}

// The whole layer on device buffers.  The host-buffer path clears the device
// status word once and runs its chunks with clear_status = false, so the
// word collects the flags of every chunk.
int forward_impl(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                 const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, void* ws,
                 size_t ws_bytes, void* stream, bool clear_status, bool two_stage_router = false) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || w_lat == nullptr || w_head == nullptr || w13 == nullptr || w_down == nullptr ||
      out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_lat) || !aligned16(w_head) || !aligned16(w13) || !aligned16(w_down) ||
      !aligned16(out) || !aligned16(ws) || (bias != nullptr && !aligned16(bias)))
    return MOE_ERR_MISALIGNED;
  const ForwardLayout f = forward_layout(dims);
  if (ws_bytes < f.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (clear_status && (rc = moe_clear_device_status(ws, stream)) != MOE_OK) return rc;
  int32_t* idx = at<int32_t>(ws, f.idx);
  float* gate = at<float>(ws, f.gate);
  int32_t* offsets = at<int32_t>(ws, f.offsets);
  int32_t* row_of = at<int32_t>(ws, f.row_of);
  int32_t* src = at<int32_t>(ws, f.src);
  moe_bf16* xperm = at<moe_bf16>(ws, f.xperm);
  moe_bf16* act = at<moe_bf16>(ws, f.act);
  // y_perm reuses x_perm's memory: x_perm is dead once expert GEMM-1 has run.
  // (moe_expert_gemm1_gather skips x_perm entirely, its A rows fetched by
  // cp.async gather warps, but on the clip workload it runs 9.8-9.9 ms
  // against 8.0-8.3 ms for GEMM-1 on x_perm plus ~1.05 ms for the gather.)
  moe_bf16* yperm = xperm;
  rc = two_stage_router
           ? moe_route_two_stage(dims, x, w_lat, w_head, bias, idx, gate, nullptr, ws, ws_bytes, stream)
           : moe_route(dims, x, w_lat, w_head, bias, idx, gate, nullptr, ws, ws_bytes, stream);
  if (rc != MOE_OK) return rc;
  if ((rc = moe_dispatch(dims, x, idx, offsets, row_of, src, xperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if ((rc = moe_expert_gemm1(dims, xperm, offsets, w13, act, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if ((rc = moe_expert_gemm2(dims, act, offsets, w_down, yperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  return moe_combine(dims, yperm, row_of, gate, out, stream);
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_STATUS: return "MOE_ERR_DEVICE_STATUS";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_check_dims(const moe_dims* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 1 || d->d < 1 || d->n_heads < 1 || d->head_dim < 1 || d->E < 1 || d->inter < 1 || d->top_k < 1)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const int64_t L = static_cast<int64_t>(d->n_heads) * d->head_dim;
  if (d->d % 64 != 0 || d->inter % 64 != 0 || L % 256 != 0 || L > (1 << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->top_k > kMaxTopK || d->top_k > d->E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->T * d->top_k >= (static_cast<int64_t>(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(d->E) * 2 * d->inter >= (static_cast<int64_t>(1) << 31) ||
      static_cast<int64_t>(d->E) * d->d >= (static_cast<int64_t>(1) << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int moe_scratch_size(const moe_dims* dims, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  const int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  *bytes = scratch_layout(dims).end;
  return MOE_OK;
}

int moe_workspace_size(const moe_dims* dims, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  const int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  *bytes = forward_layout(dims).end;
  return MOE_OK;
}

int moe_workspace_size_host(const moe_dims* dims, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  const int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  moe_dims chunk = *dims;
  chunk.T = host_one_piece(dims) ? dims->T : host_chunk_tokens(dims->T);
  const size_t io = align_up(static_cast<size_t>(dims->T) * dims->d * 2, kAlign);
  *bytes = forward_layout(&chunk).end + 2 * io;
  return MOE_OK;
}

int moe_clear_device_status(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  return cudaMemsetAsync(ws, 0, sizeof(int), static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK
                                                                                                : MOE_ERR_CUDA;
}

int moe_get_device_status(void* ws, int32_t* status, void* stream) {
  if (ws == nullptr || status == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  return v == 0 ? MOE_OK : MOE_ERR_DEVICE_STATUS;
}

int moe_selftest_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  if (ws == nullptr || limit_us == 0 || limit_us > 10000000u) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < kAlign + (128u << 10)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_selftest_timeout(at<uint16_t>(ws, kAlign), status_ptr(ws), static_cast<uint64_t>(limit_us) * 1000u,
                                 static_cast<cudaStream_t>(stream));
}

int moe_selftest_timeout_fused(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  if (ws == nullptr || limit_us == 0 || limit_us > 10000000u) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < kAlign + (96u << 10)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_ffn_fused_selftest(at<uint8_t>(ws, kAlign), status_ptr(ws), static_cast<uint64_t>(limit_us) * 1000u,
                                   static_cast<cudaStream_t>(stream));
}

int moe_prepare_weights(const moe_dims* dims, const moe_bf16* w_gate, const moe_bf16* w_up, moe_bf16* w13,
                        void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (w_gate == nullptr || w_up == nullptr || w13 == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w13)) return MOE_ERR_MISALIGNED;
  return launch_prepare_w13(w_gate, w_up, w13, dims->E, dims->inter, dims->d, static_cast<cudaStream_t>(stream));
}

int moe_route(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
              const float* bias, int32_t* topk_idx, float* topk_gate, float* logits, void* ws, size_t ws_bytes,
              void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (route_on_chip(dims))
    return moe_route_fused(dims, x, w_lat, w_head, bias, topk_idx, topk_gate, logits, ws, ws_bytes, stream);
  return moe_route_two_stage(dims, x, w_lat, w_head, bias, topk_idx, topk_gate, logits, ws, ws_bytes, stream);
}

int moe_route_two_stage(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                        const float* bias, int32_t* topk_idx, float* topk_gate, float* logits, void* ws,
                        size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || w_lat == nullptr || w_head == nullptr || topk_idx == nullptr || topk_gate == nullptr ||
      ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_lat) || !aligned16(w_head) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
      !aligned16(ws) || (bias != nullptr && !aligned16(bias)) || (logits != nullptr && !aligned16(logits)))
    return MOE_ERR_MISALIGNED;
  const ScratchLayout sl = scratch_layout(dims);
  if (ws_bytes < sl.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  RouteArgs a{};
  a.x = x;
  a.w_lat = w_lat;
  a.w_head = w_head;
  a.bias = bias;
  a.topk_idx = topk_idx;
  a.topk_gate = topk_gate;
  a.logits = logits;
  a.hl = at<uint16_t>(ws, sl.hl);
  a.T = dims->T;
  a.d = dims->d;
  a.L = dims->n_heads * dims->head_dim;
  a.E = dims->E;
  a.k = dims->top_k;
  a.head_dim = dims->head_dim;
  a.status = status_ptr(ws);
  a.sm_count = sms;
  return launch_route(a, static_cast<cudaStream_t>(stream));
}

int moe_route_fused(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                    const float* bias, int32_t* topk_idx, float* topk_gate, float* logits, void* ws, size_t ws_bytes,
                    void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (!route_fused_supported(dims->head_dim)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (x == nullptr || w_lat == nullptr || w_head == nullptr || topk_idx == nullptr || topk_gate == nullptr ||
      ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_lat) || !aligned16(w_head) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
      !aligned16(ws) || (bias != nullptr && !aligned16(bias)) || (logits != nullptr && !aligned16(logits)))
    return MOE_ERR_MISALIGNED;
  const ScratchLayout sl = scratch_layout(dims);
  if (ws_bytes < sl.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  RouteArgs a{};
  a.x = x;
  a.w_lat = w_lat;
  a.w_head = w_head;
  a.bias = bias;
  a.topk_idx = topk_idx;
  a.topk_gate = topk_gate;
  a.logits = logits;
  a.partial = at<float>(ws, sl.hl);  // [G, T, E] fp32 head-group partial scores, G * E <= L
  a.T = dims->T;
  a.d = dims->d;
  a.L = dims->n_heads * dims->head_dim;
  a.E = dims->E;
  a.k = dims->top_k;
  a.head_dim = dims->head_dim;
  a.status = status_ptr(ws);
  a.sm_count = sms;
  return launch_route_fused(a, dims->head_dim, static_cast<cudaStream_t>(stream));
}

int moe_prepare_router(const moe_dims* dims, const moe_bf16* w_lat, const moe_bf16* w_head, moe_bf16* w_router,
                       void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (w_lat == nullptr || w_head == nullptr || w_router == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_lat) || !aligned16(w_head) || !aligned16(w_router)) return MOE_ERR_MISALIGNED;
  return launch_fold_router(w_head, w_lat, dims->E, dims->n_heads * dims->head_dim, dims->d, w_router,
                            static_cast<cudaStream_t>(stream));
}

int moe_route_folded(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                     int32_t* topk_idx, float* topk_gate, float* logits, void* ws, size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || w_router == nullptr || topk_idx == nullptr || topk_gate == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) || !aligned16(ws) ||
      (bias != nullptr && !aligned16(bias)) || (logits != nullptr && !aligned16(logits)))
    return MOE_ERR_MISALIGNED;
  if (ws_bytes < scratch_layout(dims).end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  RouteArgs a{};
  a.x = x;
  a.bias = bias;
  a.topk_idx = topk_idx;
  a.topk_gate = topk_gate;
  a.logits = logits;
  a.T = dims->T;
  a.d = dims->d;
  a.L = dims->n_heads * dims->head_dim;
  a.E = dims->E;
  a.k = dims->top_k;
  a.status = status_ptr(ws);
  a.sm_count = sms;
  return launch_route_folded(a, w_router, static_cast<cudaStream_t>(stream));
}

int moe_dispatch(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx, int32_t* offsets,
                 int32_t* row_of, int32_t* src_token, moe_bf16* x_perm, void* ws, size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || topk_idx == nullptr || offsets == nullptr || row_of == nullptr || src_token == nullptr ||
      x_perm == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(offsets) || !aligned16(row_of) ||
      !aligned16(src_token) || !aligned16(x_perm) || !aligned16(ws))
    return MOE_ERR_MISALIGNED;
  const ScratchLayout sl = scratch_layout(dims);
  if (ws_bytes < sl.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  DispatchArgs a{};
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
  a.block_counts = at<int32_t>(ws, sl.disp);
  a.status = status_ptr(ws);
  a.sm_count = sms;
  return launch_dispatch(a, static_cast<cudaStream_t>(stream));
}

int moe_dispatch_indices(const moe_dims* dims, const int32_t* topk_idx, int32_t* offsets, int32_t* row_of,
                         int32_t* src_token, void* ws, size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (topk_idx == nullptr || offsets == nullptr || row_of == nullptr || src_token == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(topk_idx) || !aligned16(offsets) || !aligned16(row_of) || !aligned16(src_token) || !aligned16(ws))
    return MOE_ERR_MISALIGNED;
  const ScratchLayout sl = scratch_layout(dims);
  if (ws_bytes < sl.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  DispatchArgs a{};
  a.topk_idx = topk_idx;
  a.T = dims->T;
  a.d = dims->d;
  a.k = dims->top_k;
  a.E = dims->E;
  a.offsets = offsets;
  a.row_of = row_of;
  a.src_token = src_token;
  a.x_perm = nullptr;
  a.block_counts = at<int32_t>(ws, sl.disp);
  a.status = status_ptr(ws);
  a.sm_count = sms;
  return launch_dispatch(a, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Shared checks of the expert-GEMM entry points; fills `a` on success.
int ffn_args(const moe_dims* dims, const int32_t* offsets, void* ws, size_t ws_bytes, FfnArgs& a) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (offsets == nullptr || ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(offsets) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < scratch_layout(dims).end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  a = FfnArgs{};
  a.offsets = offsets;
  a.rows = dims->T * dims->top_k;
  a.d = dims->d;
  a.I = dims->inter;
  a.E = dims->E;
  a.status = status_ptr(ws);
  a.sm_count = sms;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_expert_gemm1(const moe_dims* dims, const moe_bf16* x_perm, const int32_t* offsets, const moe_bf16* w13,
                     moe_bf16* act, void* ws, size_t ws_bytes, void* stream) {
  FfnArgs a;
  int rc = ffn_args(dims, offsets, ws, ws_bytes, a);
  if (rc != MOE_OK) return rc;
  if (x_perm == nullptr || w13 == nullptr || act == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w13) || !aligned16(act)) return MOE_ERR_MISALIGNED;
  a.x_perm = x_perm;
  a.w13 = w13;
  a.act = act;
  return launch_gemm1(a, static_cast<cudaStream_t>(stream));
}

int moe_expert_gemm1_gather(const moe_dims* dims, const moe_bf16* x, const int32_t* src_token,
                            const int32_t* offsets, const moe_bf16* w13, moe_bf16* act, void* ws, size_t ws_bytes,
                            void* stream) {
  FfnArgs a;
  int rc = ffn_args(dims, offsets, ws, ws_bytes, a);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || src_token == nullptr || w13 == nullptr || act == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(src_token) || !aligned16(w13) || !aligned16(act)) return MOE_ERR_MISALIGNED;
  a.x = x;
  a.T = dims->T;
  a.src_token = src_token;
  a.w13 = w13;
  a.act = act;
  return launch_gemm1_gather(a, static_cast<cudaStream_t>(stream));
}

int moe_expert_gemm2(const moe_dims* dims, const moe_bf16* act, const int32_t* offsets, const moe_bf16* w_down,
                     moe_bf16* y_perm, void* ws, size_t ws_bytes, void* stream) {
  FfnArgs a;
  int rc = ffn_args(dims, offsets, ws, ws_bytes, a);
  if (rc != MOE_OK) return rc;
  if (act == nullptr || w_down == nullptr || y_perm == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(act) || !aligned16(w_down) || !aligned16(y_perm)) return MOE_ERR_MISALIGNED;
  a.act = const_cast<moe_bf16*>(act);  // read only (TMA source)
  a.w_down = w_down;
  a.y_perm = y_perm;
  return launch_gemm2(a, static_cast<cudaStream_t>(stream));
}

int moe_expert_gemm2_gated(const moe_dims* dims, const moe_bf16* act, const int32_t* offsets,
                           const moe_bf16* w_down, const int32_t* src_token, const int32_t* row_of,
                           const float* topk_gate, moe_bf16* y_perm, void* ws, size_t ws_bytes, void* stream) {
  FfnArgs a;
  int rc = ffn_args(dims, offsets, ws, ws_bytes, a);
  if (rc != MOE_OK) return rc;
  if (act == nullptr || w_down == nullptr || src_token == nullptr || row_of == nullptr || topk_gate == nullptr ||
      y_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(act) || !aligned16(w_down) || !aligned16(src_token) || !aligned16(row_of) ||
      !aligned16(topk_gate) || !aligned16(y_perm))
    return MOE_ERR_MISALIGNED;
  a.act = const_cast<moe_bf16*>(act);  // read only (TMA source)
  a.w_down = w_down;
  a.y_perm = y_perm;
  a.src_token = src_token;
  a.row_of = row_of;
  a.gate = topk_gate;
  a.T = dims->T;
  a.k = dims->top_k;
  return launch_gemm2_gated(a, static_cast<cudaStream_t>(stream));
}

int moe_expert_ffn(const moe_dims* dims, const moe_bf16* x_perm, const int32_t* offsets, const moe_bf16* w13,
                   const moe_bf16* w_down, moe_bf16* act, moe_bf16* y_perm, void* ws, size_t ws_bytes,
                   void* stream) {
  // all checks before the first launch, so a bad argument launches nothing
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x_perm == nullptr || offsets == nullptr || w13 == nullptr || w_down == nullptr || act == nullptr ||
      y_perm == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(offsets) || !aligned16(w13) || !aligned16(w_down) || !aligned16(act) ||
      !aligned16(y_perm) || !aligned16(ws))
    return MOE_ERR_MISALIGNED;
  if (ws_bytes < scratch_layout(dims).end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  rc = moe_expert_gemm1(dims, x_perm, offsets, w13, act, ws, ws_bytes, stream);
  if (rc != MOE_OK) return rc;
  return moe_expert_gemm2(dims, act, offsets, w_down, y_perm, ws, ws_bytes, stream);
}

int moe_combine(const moe_dims* dims, const moe_bf16* y_perm, const int32_t* row_of, const float* topk_gate,
                moe_bf16* out, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (y_perm == nullptr || row_of == nullptr || topk_gate == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(row_of) || !aligned16(topk_gate) || !aligned16(out))
    return MOE_ERR_MISALIGNED;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  CombineArgs a{};
  a.y_perm = y_perm;
  a.row_of = row_of;
  a.gate = topk_gate;
  a.out = out;
  a.T = dims->T;
  a.d = dims->d;
  a.k = dims->top_k;
  a.sm_count = sms;
  return launch_combine(a, static_cast<cudaStream_t>(stream));
}

int moe_combine_rows(const moe_dims* dims, const moe_bf16* y_perm, const int32_t* row_of, moe_bf16* out,
                     void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (y_perm == nullptr || row_of == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(row_of) || !aligned16(out)) return MOE_ERR_MISALIGNED;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  CombineArgs a{};
  a.y_perm = y_perm;
  a.row_of = row_of;
  a.gate = nullptr;  // rows already scaled by their gates
  a.out = out;
  a.T = dims->T;
  a.d = dims->d;
  a.k = dims->top_k;
  a.sm_count = sms;
  return launch_combine(a, static_cast<cudaStream_t>(stream));
}

int moe_forward(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, void* ws,
                size_t ws_bytes, void* stream) {
  return forward_impl(dims, x, w_lat, w_head, bias, w13, w_down, out, ws, ws_bytes, stream, true);
}

int moe_forward_fused(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                      const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, uint32_t fuse,
                      void* ws, size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if ((fuse & ~static_cast<uint32_t>(MOE_FUSE_GATHER | MOE_FUSE_GATE)) != 0u) return MOE_ERR_INVALID_ARG;
  if (x == nullptr || w_lat == nullptr || w_head == nullptr || w13 == nullptr || w_down == nullptr ||
      out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_lat) || !aligned16(w_head) || !aligned16(w13) || !aligned16(w_down) ||
      !aligned16(out) || !aligned16(ws) || (bias != nullptr && !aligned16(bias)))
    return MOE_ERR_MISALIGNED;
  const ForwardLayout f = forward_layout(dims);
  if (ws_bytes < f.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = moe_clear_device_status(ws, stream)) != MOE_OK) return rc;
  int32_t* idx = at<int32_t>(ws, f.idx);
  float* gate = at<float>(ws, f.gate);
  int32_t* offsets = at<int32_t>(ws, f.offsets);
  int32_t* row_of = at<int32_t>(ws, f.row_of);
  int32_t* src = at<int32_t>(ws, f.src);
  moe_bf16* yperm = at<moe_bf16>(ws, f.xperm);  // x_perm's region (x_perm itself not formed with the gather fused)
  moe_bf16* act = at<moe_bf16>(ws, f.act);
  if ((rc = moe_route(dims, x, w_lat, w_head, bias, idx, gate, nullptr, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if (fuse & MOE_FUSE_GATHER) {
    if ((rc = moe_dispatch_indices(dims, idx, offsets, row_of, src, ws, ws_bytes, stream)) != MOE_OK) return rc;
    rc = moe_expert_gemm1_gather(dims, x, src, offsets, w13, act, ws, ws_bytes, stream);
  } else {
    if ((rc = moe_dispatch(dims, x, idx, offsets, row_of, src, yperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
    rc = moe_expert_gemm1(dims, yperm, offsets, w13, act, ws, ws_bytes, stream);
  }
  if (rc != MOE_OK) return rc;
  if (fuse & MOE_FUSE_GATE) {
    if ((rc = moe_expert_gemm2_gated(dims, act, offsets, w_down, src, row_of, gate, yperm, ws, ws_bytes, stream)) !=
        MOE_OK)
      return rc;
    return moe_combine_rows(dims, yperm, row_of, out, stream);
  }
  if ((rc = moe_expert_gemm2(dims, act, offsets, w_down, yperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  return moe_combine(dims, yperm, row_of, gate, out, stream);
}

int moe_forward_folded(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                       const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, void* ws, size_t ws_bytes,
                       void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || w_router == nullptr || w13 == nullptr || w_down == nullptr || out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w13) || !aligned16(w_down) || !aligned16(out) ||
      !aligned16(ws) || (bias != nullptr && !aligned16(bias)))
    return MOE_ERR_MISALIGNED;
  const ForwardLayout f = forward_layout(dims);
  if (ws_bytes < f.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = moe_clear_device_status(ws, stream)) != MOE_OK) return rc;
  int32_t* idx = at<int32_t>(ws, f.idx);
  float* gate = at<float>(ws, f.gate);
  int32_t* offsets = at<int32_t>(ws, f.offsets);
  int32_t* row_of = at<int32_t>(ws, f.row_of);
  int32_t* src = at<int32_t>(ws, f.src);
  moe_bf16* xperm = at<moe_bf16>(ws, f.xperm);
  moe_bf16* act = at<moe_bf16>(ws, f.act);
  if ((rc = moe_route_folded(dims, x, w_router, bias, idx, gate, nullptr, ws, ws_bytes, stream)) != MOE_OK)
    return rc;
  if ((rc = moe_dispatch(dims, x, idx, offsets, row_of, src, xperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if ((rc = moe_expert_gemm1(dims, xperm, offsets, w13, act, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if ((rc = moe_expert_gemm2(dims, act, offsets, w_down, xperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  return moe_combine(dims, xperm, row_of, gate, out, stream);
}

}  // extern "C"

namespace {

int check_ext(const moe_dims* d, const moe_ext* x) {
  if (x == nullptr) return MOE_ERR_INVALID_ARG;
  if (x->n_shared < 0 || x->n_modalities < 0 || x->n_modalities > 8) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->top_k + x->n_shared > kMaxTopK || d->E + x->n_shared > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  for (int m = 0; m < x->n_modalities; ++m) {
    const int b = x->expert_begin[m], e = x->expert_end[m];
    if (b < 0 || e > d->E || e - b < d->top_k) return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  if (x->modality != nullptr && (reinterpret_cast<uintptr_t>(x->modality) & 3u)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_dims expanded(const moe_dims* d, const moe_ext* x) {
  moe_dims e = *d;
  e.E += x->n_shared;
  e.top_k += x->n_shared;
  return e;
}

RouteExt route_ext_of(const moe_ext* x) {
  RouteExt r{};
  r.n_shared = x->n_shared;
  r.n_mod = x->modality != nullptr ? x->n_modalities : 0;
  for (int m = 0; m < 8; ++m) {
    r.ebeg[m] = m < x->n_modalities ? x->expert_begin[m] : 0;
    r.eend[m] = m < x->n_modalities ? x->expert_end[m] : 0;
  }
  r.modality = x->modality;
  return r;
}

}  // namespace

extern "C" {

int moe_workspace_size_ext(const moe_dims* dims, const moe_ext* ext, size_t* bytes) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if ((rc = check_ext(dims, ext)) != MOE_OK) return rc;
  const moe_dims d2 = expanded(dims, ext);
  return moe_workspace_size(&d2, bytes);
}

int moe_route_ext(const moe_dims* dims, const moe_ext* ext, const moe_bf16* x, const moe_bf16* w_lat,
                  const moe_bf16* w_head, const float* bias, int32_t* topk_idx, float* topk_gate, float* logits,
                  void* ws, size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if ((rc = check_ext(dims, ext)) != MOE_OK) return rc;
  if (x == nullptr || w_lat == nullptr || w_head == nullptr || topk_idx == nullptr || topk_gate == nullptr ||
      ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_lat) || !aligned16(w_head) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
      !aligned16(ws) || (bias != nullptr && !aligned16(bias)) || (logits != nullptr && !aligned16(logits)))
    return MOE_ERR_MISALIGNED;
  const ScratchLayout sl = scratch_layout(dims);
  if (ws_bytes < sl.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count_current();
  if (sms <= 0) return MOE_ERR_CUDA;
  RouteArgs a{};
  a.x = x;
  a.w_lat = w_lat;
  a.w_head = w_head;
  a.bias = bias;
  a.topk_idx = topk_idx;
  a.topk_gate = topk_gate;
  a.logits = logits;
  a.hl = at<uint16_t>(ws, sl.hl);
  a.T = dims->T;
  a.d = dims->d;
  a.L = dims->n_heads * dims->head_dim;
  a.E = dims->E;
  a.k = dims->top_k;
  a.head_dim = dims->head_dim;
  a.ext = route_ext_of(ext);
  a.status = status_ptr(ws);
  a.sm_count = sms;
  if (route_on_chip(dims)) {  // the same choice as moe_route
    a.partial = at<float>(ws, sl.hl);
    return launch_route_fused(a, dims->head_dim, static_cast<cudaStream_t>(stream));
  }
  return launch_route(a, static_cast<cudaStream_t>(stream));
}

int moe_forward_ext(const moe_dims* dims, const moe_ext* ext, const moe_bf16* x, const moe_bf16* w_lat,
                    const moe_bf16* w_head, const float* bias, const moe_bf16* w13, const moe_bf16* w_down,
                    moe_bf16* out, void* ws, size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if ((rc = check_ext(dims, ext)) != MOE_OK) return rc;
  if (x == nullptr || w_lat == nullptr || w_head == nullptr || w13 == nullptr || w_down == nullptr ||
      out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_lat) || !aligned16(w_head) || !aligned16(w13) || !aligned16(w_down) ||
      !aligned16(out) || !aligned16(ws) || (bias != nullptr && !aligned16(bias)))
    return MOE_ERR_MISALIGNED;
  const moe_dims d2 = expanded(dims, ext);
  if ((rc = moe_check_dims(&d2)) != MOE_OK) return rc;
  const ForwardLayout f = forward_layout(&d2);
  if (ws_bytes < f.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = moe_clear_device_status(ws, stream)) != MOE_OK) return rc;
  int32_t* idx = at<int32_t>(ws, f.idx);
  float* gate = at<float>(ws, f.gate);
  int32_t* offsets = at<int32_t>(ws, f.offsets);
  int32_t* row_of = at<int32_t>(ws, f.row_of);
  int32_t* src = at<int32_t>(ws, f.src);
  moe_bf16* xperm = at<moe_bf16>(ws, f.xperm);
  moe_bf16* act = at<moe_bf16>(ws, f.act);
  if ((rc = moe_route_ext(dims, ext, x, w_lat, w_head, bias, idx, gate, nullptr, ws, ws_bytes, stream)) != MOE_OK)
    return rc;
  if ((rc = moe_dispatch(&d2, x, idx, offsets, row_of, src, xperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if ((rc = moe_expert_gemm1(&d2, xperm, offsets, w13, act, ws, ws_bytes, stream)) != MOE_OK) return rc;
  if ((rc = moe_expert_gemm2(&d2, act, offsets, w_down, xperm, ws, ws_bytes, stream)) != MOE_OK) return rc;
  return moe_combine(&d2, xperm, row_of, gate, out, stream);
}

int moe_forward_host(const moe_dims* dims, const moe_bf16* x_host, const moe_bf16* w_lat, const moe_bf16* w_head,
                     const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out_host, void* ws,
                     size_t ws_bytes, void* stream) {
  int rc = moe_check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (x_host == nullptr || out_host == nullptr || w_lat == nullptr || w_head == nullptr || w13 == nullptr ||
      w_down == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_lat) || !aligned16(w_head) || !aligned16(w13) || !aligned16(w_down) || !aligned16(ws) ||
      (bias != nullptr && !aligned16(bias)))
    return MOE_ERR_MISALIGNED;
  size_t need = 0;
  if ((rc = moe_workspace_size_host(dims, &need)) != MOE_OK) return rc;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool one_piece = host_one_piece(dims);
  const int64_t T = dims->T, tc = one_piece ? T : host_chunk_tokens(T);
  int64_t p_start[kHostPiecesMax], p_len[kHostPiecesMax];
  const int n = host_pieces(T, p_start, p_len, one_piece);
  const size_t row = static_cast<size_t>(dims->d);  // elements per token
  moe_dims cd = *dims;
  cd.T = tc;
  const size_t inner = forward_layout(&cd).end;
  const size_t io = align_up(static_cast<size_t>(T) * row * 2, kAlign);
  moe_bf16* x_dev = at<moe_bf16>(ws, inner);
  moe_bf16* out_dev = at<moe_bf16>(ws, inner + io);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  HostPipe& p = g_host_pipe[dev];
  std::lock_guard<std::mutex> lock(p.mu);
  if (!host_pipe_ready(p)) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // The copies wait for the work already queued on the caller's stream.
  bool good = ok(cudaEventRecord(p.start, s)) && ok(cudaStreamWaitEvent(p.in, p.start, 0)) &&
              ok(cudaStreamWaitEvent(p.out, p.start, 0));
  for (int i = 0; good && i < n; ++i) {
    const size_t off = static_cast<size_t>(p_start[i]) * row, bytes = static_cast<size_t>(p_len[i]) * row * 2;
    good = ok(cudaMemcpyAsync(x_dev + off, x_host + off, bytes, cudaMemcpyHostToDevice, p.in)) &&
           ok(cudaEventRecord(p.in_done[i], p.in));
  }
  if (good) rc = moe_clear_device_status(ws, stream);
  for (int i = 0; good && rc == MOE_OK && i < n; ++i) {
    const size_t off = static_cast<size_t>(p_start[i]) * row, bytes = static_cast<size_t>(p_len[i]) * row * 2;
    cd.T = p_len[i];
    good = ok(cudaStreamWaitEvent(s, p.in_done[i], 0));
    if (good)
      rc = forward_impl(&cd, x_dev + off, w_lat, w_head, bias, w13, w_down, out_dev + off, ws, inner, stream, false,
                        /*two_stage_router=*/!one_piece);
    if (good && rc == MOE_OK)
      good = ok(cudaEventRecord(p.fwd_done[i], s)) && ok(cudaStreamWaitEvent(p.out, p.fwd_done[i], 0)) &&
             ok(cudaMemcpyAsync(out_host + off, out_dev + off, bytes, cudaMemcpyDeviceToHost, p.out));
  }
  if (good) good = ok(cudaEventRecord(p.out_end, p.out)) && ok(cudaStreamWaitEvent(s, p.out_end, 0));
  // Drain all three streams, after an error too, so that no copy still uses
  // the host buffers once this returns.
  const bool in_ok = ok(cudaStreamSynchronize(p.in));
  const bool out_ok = ok(cudaStreamSynchronize(p.out));
  const bool s_ok = ok(cudaStreamSynchronize(s));
  if (rc != MOE_OK) return rc;
  return good && in_ok && out_ok && s_ok ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
