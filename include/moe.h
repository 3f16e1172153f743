/*
 * moe.h - C ABI of libmoe: forward pass of a latent-routed, top-k,
 * fine-grained SwiGLU Mixture-of-Experts layer on one NVIDIA B300 (sm_103a).
 *
 * The layer (MagiMoE as described for MAGI-2 Preview):
 *   - "MAGI-2 Preview" (heyaiwiki), Architecture table, "Routing" row and the
 *     FAQ answer "What is MagiMoE?": multi-head latent routing with 12 latent
 *     heads of 256 dims and top-6 expert selection over ultra-fine-grained
 *     experts.
 *   - "Sand.ai: The world's first 100-billion-parameter open-source MoE video
 *     generation model MAGI Preview" (36kr), section "02. Two Key Technical
 *     Decision Points": an operator library covering expert routing, sorting
 *     and calculation, fusing steps to cut intermediate results and memory
 *     traffic, tuned for many small matrix products.
 * The pages fix only the head count, head dim and top-k; the arithmetic this
 * library implements is:
 *   h      = W_lat x                              (latent projection, [L] = [n_heads*head_dim])
 *   s[e]   = sum_j <h_j, W_head[e, head j]> + b[e] (every head scores every expert; scores summed)
 *   p      = softmax(s) over all E experts
 *   idx    = the top_k experts by p, ties to the lowest expert index,
 *            slot order: p descending then index ascending
 *   gate_i = p[idx_i] / sum_j p[idx_j]
 *   y_e    = W_down[e] (silu(W_gate[e] x) * (W_up[e] x))
 *   out    = sum_i gate_i * y_{idx_i}  (slot order, fp32 accumulate, one bf16 rounding)
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, except
 *     where a name ends in _host.  The library never allocates device memory.
 *   - Matrices are row-major.  Weights are stored [out, in] ("K-major").
 *   - bf16 tensors are passed as moe_bf16 (the 16-bit pattern); fp32 as float.
 *   - Every tensor pointer and the workspace must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     enqueue work on it and return without synchronising the host, except
 *     moe_get_device_status, moe_forward_host (which ends with a stream sync)
 *     and the size queries, which launch nothing.
 *   - Arguments are checked on the host first; a failed check returns a
 *     negative moe_status and launches nothing.  A CUDA launch error returns
 *     MOE_ERR_CUDA.  Problems found on the device (an expert id outside
 *     [0, E), inconsistent group offsets, a pipeline wait that ran past its
 *     time limit) never trap: the offending row or tile is skipped and a
 *     bit is OR-ed into a sticky device status word kept in the workspace;
 *     read it with moe_get_device_status.
 *   - Shape rules: T >= 1, d % 64 == 0, inter % 64 == 0, n_heads*head_dim %
 *     256 == 0, 1 <= E <= 256, 1 <= top_k <= min(8, E), T*top_k < 2^31.
 *   - Group sizes stay on the device; no entry point reads them back, so a
 *     whole moe_forward can be enqueued without host synchronisation.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* bfloat16 bit pattern */

/* Layer dimensions.  n_heads = 12, head_dim = 256, top_k = 6 for MagiMoE. */
typedef struct moe_dims {
  int64_t T;        /* tokens in the batch */
  int32_t d;        /* hidden size */
  int32_t n_heads;  /* latent routing heads */
  int32_t head_dim; /* dims per latent head */
  int32_t E;        /* routed experts */
  int32_t inter;    /* expert intermediate size */
  int32_t top_k;    /* experts per token */
} moe_dims;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* NULL pointer, negative size, bad enum */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* dims outside the shape rules above */
  MOE_ERR_MISALIGNED = -3,         /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE_TOO_SMALL = -4,
  MOE_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_STATUS = -6,      /* moe_get_device_status found a nonzero word */
  MOE_ERR_TIMEOUT = -7             /* reserved: host-side wait gave up */
} moe_status;

/* Bits of the sticky device status word. */
#define MOE_DEV_BAD_EXPERT_ID 0x1  /* topk_idx held an id outside [0, E); that slot was skipped */
#define MOE_DEV_TIMEOUT 0x2        /* a pipeline wait exceeded its limit; that kernel stopped early */
#define MOE_DEV_BAD_OFFSETS 0x4    /* group offsets not monotone / out of range; no tile was run */
#define MOE_DEV_BAD_MODALITY 0x8   /* a token's modality id is outside [0, n_modalities); its routed slots are -1 */
#define MOE_DEV_BAD_SOURCE_ROW 0x10 /* a gathered row's src_token entry is outside [0, T); the row was read as zeros */

/* Human-readable name of a moe_status value.  Never NULL. */
const char* moe_status_string(int status);

/* Validates dims against the shape rules.  Pure host function. */
int moe_check_dims(const moe_dims* dims);

/* Bytes of scratch workspace needed by the stage calls (moe_route,
 * moe_dispatch, moe_expert_ffn): the device status word, the router's
 * latent buffer and the dispatch counters.  Pure host function. */
int moe_scratch_size(const moe_dims* dims, size_t* bytes);

/* Bytes of workspace needed by moe_forward: the scratch above plus every
 * intermediate of the layer (routing results, permutation, x_perm, act,
 * y_perm).  Any buffer of this size also serves every stage call. */
int moe_workspace_size(const moe_dims* dims, size_t* bytes);

/* Bytes of workspace needed by moe_forward_host: moe_workspace_size for one
 * token chunk of that call (see moe_forward_host) plus device staging for
 * the whole x and out. */
int moe_workspace_size_host(const moe_dims* dims, size_t* bytes);

/* Zeroes the sticky device status word in `ws` (enqueued on `stream`). */
int moe_clear_device_status(void* ws, void* stream);

/* Synchronises `stream`, then copies the device status word of `ws` to
 * *status (host).  Returns MOE_OK if it is zero, MOE_ERR_DEVICE_STATUS if
 * not (the word is left as is), MOE_ERR_CUDA if the sync failed. */
int moe_get_device_status(void* ws, int32_t* status, void* stream);

/* Self-test of device-side failure detection: runs the tensor-core GEMM
 * kernel on one tile with its loader told to issue nothing, so the kernel's
 * pipeline waits run out after limit_us microseconds (1 .. 10^7).  The
 * kernel then sets MOE_DEV_TIMEOUT in the status word of `ws`, releases its
 * tensor memory and returns; nothing faults and the context stays usable.
 * Uses the first 1 KB + 112 KB of `ws` (ws_bytes >= 129 KB).  Read the
 * result with moe_get_device_status. */
int moe_selftest_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream);

/* The same self-test for the fused head-local expert kernel (the one
 * moe_forward_headlocal runs): one 128-row tile, its weight loader told to
 * issue nothing, so the tensor-core thread's stage wait runs out after
 * limit_us microseconds (1 .. 10^7); the other roles (SwiGLU epilogue, x
 * gather) see the abort and return, tensor memory is released, and
 * MOE_DEV_TIMEOUT is set in the status word of `ws`.  Uses the first
 * 1 KB + 96 KB of `ws` (ws_bytes >= 97 KB). */
int moe_selftest_timeout_fused(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream);

/* Builds the interleaved gate/up weight used by moe_expert_ffn:
 *   w13[e] is [2*inter, d]; for block b = 0 .. inter/64 - 1 its rows
 *   [128b, 128b+64) are w_gate[e][64b, 64b+64) and rows [128b+64, 128b+128)
 *   are w_up[e][64b, 64b+64).
 * w_gate, w_up: [E, inter, d] bf16.  w13: [E, 2*inter, d] bf16 (written). */
int moe_prepare_weights(const moe_dims* dims, const moe_bf16* w_gate, const moe_bf16* w_up,
                        moe_bf16* w13, void* stream);

/* Routing (latent projection, summed head scores, softmax, top-k, gates).
 * Passage: "MAGI-2 Preview" (heyaiwiki), Architecture table, "Routing" row
 * (multi-head latent routing, 12 heads x 256 dims, top-6); the expert
 * routing step of the operator library in the 36kr article, section 02.
 *   x        [T, d] bf16
 *   w_lat    [n_heads*head_dim, d] bf16
 *   w_head   [E, n_heads*head_dim] bf16
 *   bias     [E] fp32 or NULL (added to the summed scores before the softmax)
 *   topk_idx [T, top_k] int32 (written): expert ids, slot order as above
 *   topk_gate[T, top_k] fp32 (written): renormalised gates
 *   logits   [T, E] fp32 or NULL: if given, the summed scores s (bias included)
 *   ws       scratch of at least moe_scratch_size bytes
 * The latent vector h is accumulated in fp32 on the tensor cores and fed to
 * the head-score product as a bf16 hi + lo pair, so s carries fp32-level
 * accuracy although both products run as bf16 tensor-core GEMMs.
 * Small batches (ceil(T / 128) * n_heads <= 444, three waves of B300's 148
 * SMs, and a head_dim moe_route_fused supports) take the on-chip path of
 * moe_route_fused, where h never leaves the SM; larger ones take the
 * two-stage path of moe_route_two_stage, which writes h to the workspace as
 * the bf16 pair and is faster once there are enough token tiles.  Both meet
 * the same tolerances; their last bits of s may differ. */
int moe_route(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
              const float* bias, int32_t* topk_idx, float* topk_gate, float* logits,
              void* ws, size_t ws_bytes, void* stream);

/* moe_route through the two-stage path at any size: a latent GEMM whose
 * epilogue writes h as the bf16 hi | lo pair into the workspace, then a score
 * GEMM over [h_hi | h_lo] with the softmax / top-k / gates in its epilogue. */
int moe_route_two_stage(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                        const float* bias, int32_t* topk_idx, float* topk_gate, float* logits,
                        void* ws, size_t ws_bytes, void* stream);

/* moe_route with the latent vector kept on chip: one persistent tensor-core
 * kernel accumulates each head's 128-token x head_dim block of h in tensor
 * memory (fp32), converts it to the bf16 hi/lo operand in shared memory and
 * accumulates the head scores into a second tensor-memory block; only
 * per-head-group partial scores (G x T x E fp32, G | n_heads) leave the SM,
 * summed in fixed order by a small selection kernel.  Same outputs and
 * tolerances as moe_route.  Requires head_dim % 64 == 0 and head_dim <= 256
 * (else MOE_ERR_UNSUPPORTED_SHAPE).  On B300 it is slower than moe_route
 * (2.9 vs 2.4 ms on the clip workload): the conversion of h between a head's
 * latent and score products leaves the tensor cores idle. */
int moe_route_fused(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                    const float* bias, int32_t* topk_idx, float* topk_gate, float* logits, void* ws, size_t ws_bytes,
                    void* stream);

/* Folded router (optional fast path).  The summed head scores are linear in
 * x: s = x (W_head W_lat)^T + b.  moe_prepare_router computes
 * W_eff = W_head W_lat [E, d] once per weight load (fp32 accumulation) and
 * stores it as a bf16 pair: w_router [E, 2d], row e = [bf16(W_eff[e]) |
 * bf16(W_eff[e] - hi)].  moe_route_folded then evaluates s with one bf16
 * tensor-core GEMM of K = 2d against [x | x] and applies the same bias,
 * softmax, top-k and gates as moe_route (same outputs, same tolerances);
 * the latent vector h is never formed.  Router work on the clip workload
 * drops from 2.88 to 0.23 TFLOP.  Arguments as in moe_route. */
int moe_prepare_router(const moe_dims* dims, const moe_bf16* w_lat, const moe_bf16* w_head, moe_bf16* w_router,
                       void* stream);
int moe_route_folded(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                     int32_t* topk_idx, float* topk_gate, float* logits, void* ws, size_t ws_bytes, void* stream);

/* Sorting: counting-sort permutation of the T*top_k (token, slot) pairs into
 * expert-contiguous order, then the row gather.
 * Passage: the sorting step of the operator library (routing -> sorting ->
 * calculation) in the 36kr article, section 02.
 *   topk_idx  [T, top_k] int32 (read)
 *   offsets   [E + 1] int32 (written): exclusive prefix of per-expert counts
 *   row_of    [T, top_k] int32 (written): destination row of (t, slot);
 *             the row of (t, e) is offsets[e] + #{t' < t that chose e}
 *   src_token [T*top_k] int32 (written): src_token[row_of[t, s]] = t
 *   x_perm    [T*top_k, d] bf16 (written): x_perm[r] = x[src_token[r]]
 * The result is deterministic.  An id outside [0, E) sets
 * MOE_DEV_BAD_EXPERT_ID; that pair is left out of every output. */
int moe_dispatch(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx, int32_t* offsets,
                 int32_t* row_of, int32_t* src_token, moe_bf16* x_perm,
                 void* ws, size_t ws_bytes, void* stream);

/* Calculation: grouped SwiGLU expert GEMMs over ragged expert groups.
 * Passage: the calculation step of the operator library in the 36kr article,
 * section 02 (many small matrix products, one per fine-grained expert).
 *   x_perm  [T*top_k, d] bf16, rows of expert e are [offsets[e], offsets[e+1])
 *   offsets [E + 1] int32 device array (read on the device only)
 *   w13     [E, 2*inter, d] bf16 from moe_prepare_weights
 *   w_down  [E, d, inter] bf16
 *   act     [T*top_k, inter] bf16 (written; caller-owned intermediate):
 *           silu(x W_gate^T) * (x W_up^T), fp32 accumulate, one bf16 rounding
 *   y_perm  [T*top_k, d] bf16 (written): act W_down^T, fp32 accumulate
 * y_perm may alias x_perm. */
int moe_expert_ffn(const moe_dims* dims, const moe_bf16* x_perm, const int32_t* offsets,
                   const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* act, moe_bf16* y_perm,
                   void* ws, size_t ws_bytes, void* stream);

/* The permutation of moe_dispatch without the row gather (offsets, row_of,
 * src_token only), for use with moe_expert_gemm1_gather. */
int moe_dispatch_indices(const moe_dims* dims, const int32_t* topk_idx, int32_t* offsets, int32_t* row_of,
                         int32_t* src_token, void* ws, size_t ws_bytes, void* stream);

/* moe_dispatch for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point.
 *
 * Some callers cannot call cudaMalloc or hand over a workspace: code that
 * runs inside a host framework which owns every byte of device memory and
 * forbids allocation while work is being enqueued (plugin interfaces of
 * inference runtimes), or latency-critical loops where an allocation's
 * implicit device synchronisation is not acceptable.  This variant takes no
 * workspace and allocates nothing: its counters live in a fixed array inside
 * libmoe's device image, 64 + 65536 int32 (about 256 KiB), which every GPU
 * that loads the library holds until the process exits.
 *   - Arguments and results as in moe_dispatch (same kernels, same output).
 *   - status: optional device int32 that receives MOE_DEV_* bits (OR-ed in;
 *     the caller clears it).  NULL: device-detected problems are not reported.
 *   - Limit: ceil(T / 2048) * E <= 65536 (e.g. T <= 1,048,576 at E = 128);
 *     larger problems return MOE_ERR_UNSUPPORTED_SHAPE and launch nothing.
 *   - Every call looks up the array's address in the current context
 *     (cudaGetSymbolAddress, which allocates nothing), so the entry point
 *     stays correct after a cudaDeviceReset or under another context on the
 *     same device.  The first call in a context also loads the library's
 *     device code there: make that first call before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents.  Every counter is rewritten before it is read, so nothing
 *     needs clearing, but calls that overlap on the GPU (different streams,
 *     or host threads enqueueing concurrently) race on it: serialise them. */
int moe_dispatch_noalloc(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx, int32_t* offsets,
                         int32_t* row_of, int32_t* src_token, moe_bf16* x_perm, int32_t* status, void* stream);

/* The two halves of moe_expert_ffn, for callers that schedule or time them
 * separately.  moe_expert_gemm1 writes act = silu(x W_gate^T) * (x W_up^T);
 * moe_expert_gemm2 writes y_perm = act W_down^T.  Arguments as in
 * moe_expert_ffn. */
int moe_expert_gemm1(const moe_dims* dims, const moe_bf16* x_perm, const int32_t* offsets, const moe_bf16* w13,
                     moe_bf16* act, void* ws, size_t ws_bytes, void* stream);
/* moe_expert_gemm1 with the sorting gather fused into the operand loads:
 * row r of the A operand is x[src_token[r]] (x [T, d], src_token from
 * moe_dispatch / moe_dispatch_indices), fetched with 16-byte asynchronous
 * copies by four extra warps of the GEMM kernel, so x_perm is never
 * materialised (saves T*top_k*d*2 bytes of memory and the gather's HBM round
 * trip).  The result equals moe_expert_gemm1 on the gathered x_perm bit for
 * bit.  moe_forward_fused with MOE_FUSE_GATHER runs it; on B300 the gathered
 * GEMM-1 takes ~1.12x the time of moe_expert_gemm1 on x_perm, about what the
 * separate gather costs, so that layer and moe_forward run at the same speed
 * on the clip workload; moe_forward keeps the separate gather.  A src_token
 * entry outside [0, T) is not dereferenced: that row reads as zeros and
 * MOE_DEV_BAD_SOURCE_ROW is set in the status word of `ws`. */
int moe_expert_gemm1_gather(const moe_dims* dims, const moe_bf16* x, const int32_t* src_token,
                            const int32_t* offsets, const moe_bf16* w13, moe_bf16* act, void* ws, size_t ws_bytes,
                            void* stream);
int moe_expert_gemm2(const moe_dims* dims, const moe_bf16* act, const int32_t* offsets, const moe_bf16* w_down,
                     moe_bf16* y_perm, void* ws, size_t ws_bytes, void* stream);

/* Gate-weighted combine, scatter-free (one writer per output row).
 * Passage: the end of the routing -> sorting -> calculation chain in the
 * 36kr article, section 02 (expert outputs brought back to token order and
 * summed with the router's weights):
 *   out[t] = sum_{s < top_k} topk_gate[t, s] * y_perm[row_of[t, s]]
 * summed in slot order in fp32, rounded once to bf16.  A row index outside
 * [0, T*top_k) contributes nothing.
 *   y_perm [T*top_k, d] bf16, row_of [T, top_k] int32, topk_gate [T, top_k] fp32,
 *   out [T, d] bf16 (written). */
int moe_combine(const moe_dims* dims, const moe_bf16* y_perm, const int32_t* row_of,
                const float* topk_gate, moe_bf16* out, void* stream);

/* The whole layer: moe_route, moe_dispatch, moe_expert_ffn, moe_combine on
 * one stream, intermediates in `ws` (at least moe_workspace_size bytes).
 * Passage: MagiMoE in "MAGI-2 Preview" (heyaiwiki), FAQ "What is MagiMoE?",
 * and the operator library of the 36kr article, section 02.
 * Clears the device status word first.  Weights: w13 from
 * moe_prepare_weights, w_down [E, d, inter]. */
int moe_forward(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out,
                void* ws, size_t ws_bytes, void* stream);

/* Fusions of the layer's steps (the 36kr article, section 02: the operator
 * library fuses calculation steps to cut intermediate results and memory
 * traffic).
 *
 * moe_expert_gemm2_gated: moe_expert_gemm2 with the gate multiply in its
 * epilogue, y_perm[r] = bf16(topk_gate[t, s] * (act W_down^T)[r]) where
 * t = src_token[r] and row_of[t, s] = r (so y is rounded to bf16 after the
 * gate, not before).  src_token, row_of: from moe_dispatch; topk_gate from
 * moe_route.  A row whose token does not list it gets gate 0.
 *
 * moe_combine_rows: out[t] = sum_{s < top_k} y_perm[row_of[t, s]] (rows
 * already scaled by their gates), fp32 sum in slot order, one bf16 rounding.
 *
 * moe_forward_fused: moe_forward with a choice of fusions (fuse = OR of):
 *   MOE_FUSE_GATHER  the sorting gather runs inside expert GEMM-1's operand
 *                    loads (moe_dispatch_indices + moe_expert_gemm1_gather):
 *                    x_perm is never written or read back
 *   MOE_FUSE_GATE    the gate multiply runs in expert GEMM-2's epilogue
 *                    (moe_expert_gemm2_gated + moe_combine_rows)
 * fuse = 0 is moe_forward's sequence.  Unknown bits: MOE_ERR_INVALID_ARG.
 * Same workspace as moe_forward; same outputs within the layer's
 * tolerances (with MOE_FUSE_GATE the bf16 rounding of y_perm moves after
 * the gate, so the bits differ from moe_forward's). */
#define MOE_FUSE_GATHER 0x1u
#define MOE_FUSE_GATE 0x2u
int moe_expert_gemm2_gated(const moe_dims* dims, const moe_bf16* act, const int32_t* offsets,
                           const moe_bf16* w_down, const int32_t* src_token, const int32_t* row_of,
                           const float* topk_gate, moe_bf16* y_perm, void* ws, size_t ws_bytes, void* stream);
int moe_combine_rows(const moe_dims* dims, const moe_bf16* y_perm, const int32_t* row_of, moe_bf16* out,
                     void* stream);
int moe_forward_fused(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_lat, const moe_bf16* w_head,
                      const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, uint32_t fuse,
                      void* ws, size_t ws_bytes, void* stream);

/* moe_forward with the folded router (w_router from moe_prepare_router). */
int moe_forward_folded(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                       const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, void* ws, size_t ws_bytes,
                       void* stream);

/* Shared and modality-specific experts (36kr article, section 02: shared
 * experts carry what the modalities have in common, modality-specific
 * experts what is unique to language, picture or sound).  The E routed
 * experts are split into per-modality ranges [expert_begin[m], expert_end[m]);
 * a token of modality m is routed only within its range (softmax, top-k and
 * renormalised gates over those experts).  n_shared shared experts, stored
 * after the routed ones in w13/w_down (ids E .. E+n_shared-1), process every
 * token with weight 1:
 *   out[t] = sum_i gate[t,i] FFN_{idx[t,i]}(x[t]) + sum_j FFN_{E+j}(x[t])
 * Rules: n_shared >= 0, top_k + n_shared <= 8, E + n_shared <= 256,
 * 0 <= n_modalities <= 8 (0: no masking), each range inside [0, E) with at
 * least top_k experts.  modality: device int32 [T] (4-byte aligned), or NULL
 * for no masking; an id outside [0, n_modalities) sets MOE_DEV_BAD_MODALITY
 * and leaves that token's routed slots at -1. */
typedef struct moe_ext {
  int32_t n_shared;
  int32_t n_modalities;
  int32_t expert_begin[8];
  int32_t expert_end[8];
  const int32_t* modality;
} moe_ext;

/* Workspace for moe_forward_ext (= moe_workspace_size with E + n_shared
 * experts and top_k + n_shared slots). */
int moe_workspace_size_ext(const moe_dims* dims, const moe_ext* ext, size_t* bytes);

/* Routing with modality ranges; writes top_k + n_shared slots per token
 * (topk_idx/topk_gate [T, top_k + n_shared]: the routed slots, then the
 * shared experts with gate 1).  logits [T, E] (optional) are the unmasked
 * summed scores.  Other arguments, and the choice between the on-chip and
 * the two-stage path, as in moe_route. */
int moe_route_ext(const moe_dims* dims, const moe_ext* ext, const moe_bf16* x, const moe_bf16* w_lat,
                  const moe_bf16* w_head, const float* bias, int32_t* topk_idx, float* topk_gate, float* logits,
                  void* ws, size_t ws_bytes, void* stream);

/* The whole layer with modality ranges and shared experts.  w13
 * [E + n_shared, 2*inter, d] (moe_prepare_weights with E + n_shared experts),
 * w_down [E + n_shared, d, inter]; ws: moe_workspace_size_ext bytes. */
int moe_forward_ext(const moe_dims* dims, const moe_ext* ext, const moe_bf16* x, const moe_bf16* w_lat,
                    const moe_bf16* w_head, const float* bias, const moe_bf16* w13, const moe_bf16* w_down,
                    moe_bf16* out, void* ws, size_t ws_bytes, void* stream);

/* Head-local MultiHead MoE (36kr article, section 02: the hidden
 * representation split into heads, each head choosing its own experts in its
 * own low-dimensional subspace, the head results fused back).  Here
 * dims->d = n_heads * head_dim and dims->E is the number of experts PER
 * HEAD; head j's slice x_j = x[:, j*head_dim : (j+1)*head_dim] is scored by
 * its own router, s_j = x_j W_router[j]^T + bias[j], softmax, top_k (ties
 * to the lowest index), renormalised gates; its chosen head-local SwiGLU
 * experts (head_dim -> inter -> head_dim) are combined into out's columns
 * of head j (concatenation of the heads).
 *   w_router [n_heads, E, head_dim] bf16, bias [n_heads, E] fp32 or NULL
 *   w13 [n_heads, E, 2*inter, head_dim] from moe_prepare_weights_headlocal
 *   w_down [n_heads, E, head_dim, inter] bf16, out [T, d] bf16
 *   topk_idx [n_heads, T, top_k] int32 or NULL (written: each head's choice)
 *   logits [n_heads, T, E] fp32 or NULL (written: each head's scores)
 * Rules: head_dim % 64 == 0, inter % 64 == 0, E <= 256, top_k <= min(8, E).
 * All heads' routers run as one batched GEMM, their sorts and combines as
 * single launches over (head, token), all on `stream`.  With head_dim <= 256
 * and inter a multiple of 128, both expert layers of all n_heads * E
 * head-local experts run as one fused kernel: it copies each 128-row tile's
 * x head slices from x by source token into shared memory (no sorted copy of
 * x is written) and keeps the tile's activations on chip (the gate/up
 * products in tensor memory, SwiGLU into shared memory, the down projection
 * accumulating in tensor memory), so neither x_perm nor act reaches HBM.
 * moe_forward_headlocal_staged runs the same layer with a separate gather
 * and the two expert layers as separate grouped GEMMs (x_perm and act
 * through the workspace; head by head when n_heads * E > 3072); both give
 * the same bits. */
int moe_workspace_size_headlocal(const moe_dims* dims, size_t* bytes);
int moe_prepare_weights_headlocal(const moe_dims* dims, const moe_bf16* w_gate, const moe_bf16* w_up, moe_bf16* w13,
                                  void* stream);
int moe_forward_headlocal(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                          const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out, int32_t* topk_idx,
                          float* logits, void* ws, size_t ws_bytes, void* stream);
int moe_forward_headlocal_staged(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_router,
                                 const float* bias, const moe_bf16* w13, const moe_bf16* w_down, moe_bf16* out,
                                 int32_t* topk_idx, float* logits, void* ws, size_t ws_bytes, void* stream);

/* moe_forward for a caller whose activations live in host memory: x_host
 * [T, d] in, out_host [T, d] out, weights on the device; returns after the
 * result is in out_host (the call synchronises `stream`).  The layer runs
 * over n = min(ceil(T / 8192), 8) token chunks of ceil(T / n) tokens (for
 * n >= 3 the first and last chunk are cut 1:3, the short piece at the end of
 * the batch): the chunks' copies to the device run on one internal stream
 * and the copies back on another, overlapping the compute of the
 * neighbouring chunks on `stream`.  A batch that moe_route would route on
 * chip runs as one piece; otherwise every piece takes the two-stage router.
 * Each token's result has the same bits as moe_forward over the whole
 * batch.  The device status word at the start of ws collects the flags
 * of every chunk.  Host buffers should be page-locked: pageable memory still
 * gives correct results, but the copies then serialise with the compute.
 * Calls for the same device are serialised by an internal lock.  ws: at
 * least moe_workspace_size_host bytes. */
int moe_forward_host(const moe_dims* dims, const moe_bf16* x_host, const moe_bf16* w_lat,
                     const moe_bf16* w_head, const float* bias, const moe_bf16* w13,
                     const moe_bf16* w_down, moe_bf16* out_host, void* ws, size_t ws_bytes,
                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
