// Head-local MultiHead MoE: the hidden vector (d = n_heads * head_dim) is split
// into head slices; head j routes its own slice over its own E experts (router
// GEMM + fused top-k), sorts its tokens, runs its head-local SwiGLU experts
// (head_dim -> inter -> head_dim, grouped tcgen05 GEMMs) and combines into its
// head_dim columns of out.  All heads go through each stage together: one
// batched router GEMM, one sort/gather over (head, token), one grouped GEMM
// per expert layer over all n_heads * E head-local experts (head by head only
// when they exceed the engine's group table), one combine.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "internal.h"
#include "moe.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 1024;
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_hl(const moe_dims* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 1 || d->n_heads < 1 || d->head_dim < 1 || d->E < 1 || d->inter < 1 || d->top_k < 1)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(d->n_heads) * d->head_dim != d->d) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->head_dim % 64 != 0 || d->inter % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->E > kMaxExperts || d->top_k > kMaxTopK || d->top_k > d->E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->T * d->top_k >= (static_cast<int64_t>(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(d->n_heads) * d->E * 2 * d->inter >= (static_cast<int64_t>(1) << 31) ||
      static_cast<int64_t>(d->n_heads) * d->E * d->head_dim >= (static_cast<int64_t>(1) << 31) ||
      static_cast<int64_t>(d->n_heads) * d->T * d->top_k >= (static_cast<int64_t>(1) << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

struct HlLayout {
  size_t disp, idx, gate, offsets, goff, tiles, row_of, src, xperm, act, end;
};

// Per-head arrays side by side: idx/gate/row_of/src [H, T, k], offsets [H, E+1],
// y_perm [H, T*k, head_dim] (the staged path's x_perm first), act [H, T*k,
// inter] (staged path only), dispatch
// counters [H][nblk][E]; goff [H*E + 1]: the group offsets of all heads'
// experts over the concatenated rows (head h's rows start at h*T*k); tiles
// [H*E + 1]: the fused expert kernel's table of the groups' tile counts.
HlLayout hl_layout(const moe_dims* d) {
  HlLayout l;
  const size_t H = d->n_heads;
  const size_t Tk = static_cast<size_t>(d->T) * d->top_k;
  l.disp = kAlign;
  l.idx = align_up(l.disp + H * dispatch_scratch_bytes(d->T, d->E), kAlign);
  l.gate = align_up(l.idx + H * Tk * 4, kAlign);
  l.offsets = align_up(l.gate + H * Tk * 4, kAlign);
  l.goff = align_up(l.offsets + H * (static_cast<size_t>(d->E) + 1) * 4, kAlign);
  l.tiles = align_up(l.goff + (H * d->E + 1) * 4, kAlign);
  l.row_of = align_up(l.tiles + (H * d->E + 1) * 4, kAlign);
  l.src = align_up(l.row_of + H * Tk * 4, kAlign);
  l.xperm = align_up(l.src + H * Tk * 4, kAlign);
  l.act = align_up(l.xperm + H * Tk * d->head_dim * 2, kAlign);
  l.end = align_up(l.act + H * Tk * d->inter * 2, kAlign);
  return l;
}

// goff[h*E + e] = h*Tk + offsets[h][e], goff[H*E] = H*Tk.
__global__ void concat_offsets_kernel(const int32_t* __restrict__ offsets, int H, int E, int64_t Tk,
                                      int32_t* __restrict__ goff) {
  const int64_t n = static_cast<int64_t>(H) * E;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i <= n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t h = i / E, e = i - h * E;
    goff[i] = static_cast<int32_t>(i == n ? H * Tk : h * Tk + offsets[h * (E + 1) + e]);
  }
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

extern "C" {

int moe_workspace_size_headlocal(const moe_dims* dims, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  const int rc = check_hl(dims);
  if (rc != MOE_OK) return rc;
  *bytes = hl_layout(dims).end;
  return MOE_OK;
}

int moe_prepare_weights_headlocal(const moe_dims* dims, const moe_bf16* w_gate, const moe_bf16* w_up, moe_bf16* w13,
                                  void* stream) {
  int rc = check_hl(dims);
  if (rc != MOE_OK) return rc;
  if (w_gate == nullptr || w_up == nullptr || w13 == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w13)) return MOE_ERR_MISALIGNED;
  // the n_heads * E head-local experts interleave exactly like E experts of width head_dim
  return launch_prepare_w13(w_gate, w_up, w13, dims->n_heads * dims->E, dims->inter, dims->head_dim,
                            static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// The head-local layer; `staged` runs the two expert GEMMs as separate
// grouped GEMMs (act through HBM) instead of the fused expert kernel.
int forward_headlocal(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                      const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, int32_t* topk_idx, float* logits,
                      void* ws, size_t ws_bytes, void* stream, bool staged) {
  int rc = check_hl(dims);
  if (rc != MOE_OK) return rc;
  if (x == nullptr || w_router == nullptr || w13 == nullptr || w_down == nullptr || out == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w13) || !aligned16(w_down) || !aligned16(out) ||
      !aligned16(ws) || (bias != nullptr && !aligned16(bias)) || (topk_idx != nullptr && !aligned16(topk_idx)) ||
      (logits != nullptr && !aligned16(logits)))
    return MOE_ERR_MISALIGNED;
  const HlLayout l = hl_layout(dims);
  if (ws_bytes < l.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = moe_clear_device_status(ws, stream)) != MOE_OK) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return MOE_ERR_CUDA;

  const int H = dims->n_heads, Dh = dims->head_dim, E = dims->E, I = dims->inter, k = dims->top_k;
  const int64_t T = dims->T, Tk = T * k;
  int* status = static_cast<int*>(ws);
  int32_t* idx = topk_idx != nullptr ? topk_idx : at<int32_t>(ws, l.idx);
  float* gate = at<float>(ws, l.gate);

  // 1. every head's router in one batched GEMM (fused top-k)
  rc = launch_router_headlocal(x, T, dims->d, H, Dh, w_router, E, k, bias, idx, gate, logits, status, sms, s);
  if (rc != MOE_OK) return rc;

  // 2. every head's sort and gather in one set of launches
  DispatchArgs da{};
  da.x = x;
  da.x_ld = dims->d;
  da.x_head_off = Dh;
  da.heads = H;
  da.topk_idx = idx;
  da.T = T;
  da.d = Dh;
  da.k = k;
  da.E = E;
  da.offsets = at<int32_t>(ws, l.offsets);
  da.row_of = at<int32_t>(ws, l.row_of);
  da.src_token = at<int32_t>(ws, l.src);
  const bool fused = !staged && ffn_fused_supported(Dh, I);
  // the fused expert kernel gathers its x rows itself: the sort is indices only
  da.x_perm = fused ? nullptr : at<uint16_t>(ws, l.xperm);
  da.block_counts = at<int32_t>(ws, l.disp);
  da.status = status;
  da.sm_count = sms;
  if ((rc = launch_dispatch(da, s)) != MOE_OK) return rc;

  // 3. both expert layers over all heads' experts at once (group h*E + e =
  //    expert e of head h): the fused kernel (x gathered on chip, act on
  //    chip), or the two grouped GEMMs (y_perm overwrites x_perm), head by
  //    head when the n_heads * E groups exceed the engine's table
  FfnArgs fa{};
  fa.d = Dh;
  fa.I = I;
  fa.status = status;
  fa.sm_count = sms;
  uint16_t* act = at<uint16_t>(ws, l.act);
  if (fused || static_cast<int64_t>(H) * E <= kMaxGemmGroups) {
    int32_t* goff = at<int32_t>(ws, l.goff);
    const int64_t n = static_cast<int64_t>(H) * E + 1;
    const int blocks = static_cast<int>((n + 255) / 256 < sms ? (n + 255) / 256 : sms);
    concat_offsets_kernel<<<blocks, 256, 0, s>>>(da.offsets, H, E, Tk, goff);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    fa.offsets = goff;
    fa.rows = static_cast<int64_t>(H) * Tk;
    fa.E = H * E;
    fa.x_perm = da.x_perm;
    fa.w13 = w13;
    fa.w_down = w_down;
    fa.y_perm = at<uint16_t>(ws, l.xperm);  // x_perm's region (staged: x_perm is dead once GEMM-1 has read it)
    if (fused) {  // both expert layers in one kernel, x gathered on chip, act never leaves the SM
      fa.x = x;
      fa.x_ld = dims->d;
      fa.src_token = da.src_token;
      fa.T = T;
      fa.head_groups = E;
      fa.tiles = at<int32_t>(ws, l.tiles);
      if ((rc = launch_ffn_fused(fa, s)) != MOE_OK) return rc;
    } else {
      fa.act = act;
      if ((rc = launch_gemm1(fa, s)) != MOE_OK) return rc;
      if ((rc = launch_gemm2(fa, s)) != MOE_OK) return rc;
    }
  } else {
    for (int j = 0; j < H; ++j) {
      fa.offsets = da.offsets + static_cast<int64_t>(j) * (E + 1);
      fa.rows = Tk;
      fa.E = E;
      fa.x_perm = da.x_perm + static_cast<int64_t>(j) * Tk * Dh;
      fa.w13 = w13 + static_cast<int64_t>(j) * E * 2 * I * Dh;
      fa.act = act + static_cast<int64_t>(j) * Tk * I;
      if ((rc = launch_gemm1(fa, s)) != MOE_OK) return rc;
      fa.w_down = w_down + static_cast<int64_t>(j) * E * Dh * I;
      fa.y_perm = da.x_perm + static_cast<int64_t>(j) * Tk * Dh;
      if ((rc = launch_gemm2(fa, s)) != MOE_OK) return rc;
    }
  }

  // 4. every head's combine into its columns of out, one launch
  CombineArgs ca{};
  ca.y_perm = at<uint16_t>(ws, l.xperm);
  ca.row_of = da.row_of;
  ca.gate = gate;
  ca.out = out;
  ca.out_ld = dims->d;
  ca.heads = H;
  ca.T = T;
  ca.d = Dh;
  ca.k = k;
  ca.sm_count = sms;
  return launch_combine(ca, s);
}

}  // namespace

extern "C" {

int moe_forward_headlocal(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                          const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, int32_t* topk_idx,
                          float* logits, void* ws, size_t ws_bytes, void* stream) {
  return forward_headlocal(dims, x, w_router, bias, w13, w_down, out, topk_idx, logits, ws, ws_bytes, stream,
                           false);
}

int moe_forward_headlocal_staged(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router,
                                 const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out,
                                 int32_t* topk_idx, float* logits, void* ws, size_t ws_bytes, void* stream) {
  return forward_headlocal(dims, x, w_router, bias, w13, w_down, out, topk_idx, logits, ws, ws_bytes, stream,
                           true);
}

}  // extern "C"
