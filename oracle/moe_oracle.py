"""fp64 CPU oracle for the latent-routed top-k SwiGLU MoE layer forward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its Python binding) never calls it, and it shares no code
with that path: it reads the same seeded bf16 bit patterns and nothing else.

What it computes follows the pages' description of MagiMoE:

* "MAGI-2 Preview" (heyaiwiki), Architecture table, rows "Architecture" and
  "Routing", and the FAQ answer "What is MagiMoE?": multi-head latent routing,
  12 latent heads x 256 dims, top-6 selection.
* "Sand.ai: The world's first 100-billion-parameter open-source MoE video
  generation model MAGI Preview" (36kr), section "02. Two Key Technical
  Decision Points": the operator chain routing -> sorting -> calculation over
  many small expert matrices.

The pages leave the arithmetic open; the readings taken (one learned latent
projection, every head scores every expert, head scores summed, softmax over
all experts, top-k with ties to the lowest expert index, gates renormalised
over the chosen set, SwiGLU experts, gate-weighted sum) are listed with the
reasons in the design notes.  Every step is done in float64 with no
intermediate rounding; bf16 inputs are widened exactly.

Parity: every function below is pinned by ``tests/test_oracle_pins.py``
(hand-worked example, brute-force top-k, closed forms, invariants and
planted-mistake checks).
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit


# ----------------------------------------------------------------------------
# input widening
# ----------------------------------------------------------------------------

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly.

    A bf16 value is the upper half of an IEEE float32; shifting the 16 bits
    into the high half gives that float32, and float32 -> float64 is exact.
    """
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# routing (MAGI-2 Preview Architecture table "Routing" row; FAQ "What is MagiMoE?")
# ----------------------------------------------------------------------------

def latent_projection(x: np.ndarray, w_lat: np.ndarray) -> np.ndarray:
    """h[t, :] = W_lat @ x[t]: each token's hidden vector projected to the
    n_heads x head_dim latent space (12 x 256 in MAGI-2 Preview).

    x [T, d], w_lat [n_heads*head_dim, d] -> h [T, n_heads*head_dim]; head j
    owns columns [j*head_dim, (j+1)*head_dim).
    """
    return x @ w_lat.T


def head_scores(h: np.ndarray, w_head: np.ndarray, bias, n_heads: int, head_dim: int) -> np.ndarray:
    """Summed head scores s[t, e] = sum_j <h[t, head j], W_head[e, head j]> + b[e].

    Each latent head scores every expert with its own slice of W_head
    [E, n_heads*head_dim]; the per-head scores are added.  The router bias
    (zero when None) is added once to the sum, before the softmax.
    """
    T = h.shape[0]
    E = w_head.shape[0]
    s = np.zeros((T, E), dtype=np.float64)
    for j in range(n_heads):
        cols = slice(j * head_dim, (j + 1) * head_dim)
        s += h[:, cols] @ w_head[:, cols].T
    if bias is not None:
        s += np.asarray(bias, dtype=np.float64)[None, :]
    return s


def softmax(s: np.ndarray) -> np.ndarray:
    """Row softmax over all experts: p = exp(s - max) / sum exp(s - max)."""
    z = s - s.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=1, keepdims=True)


def topk_select(p: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row, ties to the lowest index.

    Slot order: value descending, then expert index ascending.  A stable sort
    on -p keeps equal values in index order, so the lowest index wins a tie.
    Applied to the scores s (or to softmax(s): the same indices, as exp is
    monotone; s keeps values distinct where exp would underflow to 0).
    """
    order = np.argsort(-p, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def renormalised_gates(p: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """gate[t, i] = p[t, idx[t, i]] / sum_j p[t, idx[t, j]]."""
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route(x, w_lat, w_head, bias, n_heads: int, head_dim: int, k: int):
    """Latent routing: returns (logits s [T,E], topk_idx [T,k], gates [T,k])."""
    h = latent_projection(x, w_lat)
    s = head_scores(h, w_head, bias, n_heads, head_dim)
    p = softmax(s)
    idx = topk_select(s, k)   # the k largest p are the k largest s (exp is monotone)
    return s, idx, renormalised_gates(p, idx)


# ----------------------------------------------------------------------------
# sorting: tokens into expert-contiguous order (36kr, section 02, operator
# library "routing, sorting and calculation")
# ----------------------------------------------------------------------------

def dispatch(topk_idx: np.ndarray, E: int):
    """Counting-sort permutation of the (token, slot) assignments.

    count[e]  = number of (t, s) with topk_idx[t, s] == e
    offsets   = exclusive prefix sum of count, length E + 1
    row of (t, s) = offsets[e] + number of tokens t' < t that also chose e
    src_token[row] = t.

    Returns (counts [E], offsets [E+1], row_of [T,k], src_token [T*k]), all
    int64.  Raises ValueError on an expert id outside [0, E).
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    if idx.size and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.ravel():
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = np.zeros(E, dtype=np.int64)
    row_of = np.zeros((T, k), dtype=np.int64)
    src_token = np.zeros(T * k, dtype=np.int64)
    for t in range(T):
        for s in range(k):
            e = idx[t, s]
            r = offsets[e] + fill[e]
            fill[e] += 1
            row_of[t, s] = r
            src_token[r] = t
    return counts, offsets, row_of, src_token


def gather(x: np.ndarray, src_token: np.ndarray) -> np.ndarray:
    """x_perm[r] = x[src_token[r]]."""
    return x[np.asarray(src_token, dtype=np.int64)]


# ----------------------------------------------------------------------------
# calculation: SwiGLU experts and the gate-weighted combine
# ----------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z)."""
    return z * expit(z)


def expert_ffn(x_perm, offsets, w_gate, w_up, w_down, widen=None) -> np.ndarray:
    """y_perm rows of expert e: (silu(x W_gate[e]^T) * (x W_up[e]^T)) W_down[e]^T.

    x_perm [R, d] (float64), offsets [E+1]; w_gate/w_up [E, inter, d],
    w_down [E, d, inter].  If ``widen`` is given the weights are bf16 bit
    arrays and each expert's matrices are widened when that expert runs.
    """
    R, d = x_perm.shape
    E = len(offsets) - 1
    y = np.zeros((R, w_down.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        wg, wu, wd = w_gate[e], w_up[e], w_down[e]
        if widen is not None:
            wg, wu, wd = widen(wg), widen(wu), widen(wd)
        rows = x_perm[lo:hi]
        g = rows @ wg.T
        u = rows @ wu.T
        act = silu(g) * u
        y[lo:hi] = act @ wd.T
    return y


def combine(y_perm: np.ndarray, row_of: np.ndarray, gates: np.ndarray) -> np.ndarray:
    """out[t] = sum over slots s (in slot order) of gates[t,s] * y_perm[row_of[t,s]]."""
    T, k = row_of.shape
    out = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    for s in range(k):
        out += gates[:, s:s + 1] * y_perm[np.asarray(row_of[:, s], dtype=np.int64)]
    return out


# ----------------------------------------------------------------------------
# whole layer
# ----------------------------------------------------------------------------

def forward(x, w_lat, w_head, bias, w_gate, w_up, w_down, n_heads, head_dim, k,
            topk_idx=None, widen_experts=None):
    """The layer forward in float64.

    All array arguments are float64 except when ``widen_experts`` is given,
    in which case the expert weights are bf16 bits widened per expert.  If
    ``topk_idx`` is given the routing decision is taken from it (the gates are
    still the oracle's own softmax over its own logits, renormalised over that
    set); otherwise the oracle's own top-k is used.

    Returns a dict with logits, topk_idx, gates, counts, offsets, row_of,
    src_token, y_perm and out.
    """
    s = head_scores(latent_projection(x, w_lat), w_head, bias, n_heads, head_dim)
    p = softmax(s)
    # select on s: same set as on p, and exp underflow cannot turn distinct
    # scores into ties
    idx = topk_select(s, k) if topk_idx is None else np.asarray(topk_idx, dtype=np.int32)
    gates = renormalised_gates(p, idx)
    counts, offsets, row_of, src_token = dispatch(idx, w_head.shape[0])
    x_perm = gather(x, src_token)
    y_perm = expert_ffn(x_perm, offsets, w_gate, w_up, w_down, widen=widen_experts)
    out = combine(y_perm, row_of, gates)
    return dict(logits=s, topk_idx=idx, gates=gates, counts=counts, offsets=offsets,
                row_of=row_of, src_token=src_token, y_perm=y_perm, out=out)


# ----------------------------------------------------------------------------
# shared and modality-specific experts (36kr, section 02: shared experts carry
# what the modalities have in common, modality-specific experts the parts
# unique to text, picture or sound)
# ----------------------------------------------------------------------------

def modality_mask(modality, expert_ranges, E):
    """allowed[t, e]: routed expert e lies in the range of token t's modality.

    expert_ranges[m] = (begin, end) of modality m's routed experts; with no
    ranges every expert is allowed.
    """
    T = len(modality)
    if not expert_ranges:
        return np.ones((T, E), dtype=bool)
    allowed = np.zeros((T, E), dtype=bool)
    for t in range(T):
        b, e = expert_ranges[int(modality[t])]
        allowed[t, b:e] = True
    return allowed


def swiglu_ffn(x, wg, wu, wd):
    """One SwiGLU expert applied to every row: (silu(x wg^T) * (x wu^T)) wd^T."""
    return (silu(x @ wg.T) * (x @ wu.T)) @ wd.T


def forward_ext(x, w_lat, w_head, bias, w_gate, w_up, w_down, n_heads, head_dim, k, modality=None,
                expert_ranges=(), n_shared=0, topk_idx=None, widen_experts=None):
    """Layer with modality-specific routed experts and shared experts.

    Routed experts are 0 .. E-1 (E = rows of w_head); a token of modality m is
    routed only among experts [begin_m, end_m): the softmax runs over those
    experts, the top-k is taken among them and the gates are renormalised over
    the chosen k.  Experts E .. E+n_shared-1 of w_gate/w_up/w_down are shared:
    every token passes through each of them with weight 1.
        out[t] = sum_i gate[t,i] * FFN_{idx[t,i]}(x[t]) + sum_j FFN_{E+j}(x[t])
    """
    E = w_head.shape[0]
    T = x.shape[0]
    s = head_scores(latent_projection(x, w_lat), w_head, bias, n_heads, head_dim)
    modality = np.zeros(T, dtype=np.int64) if modality is None else np.asarray(modality)
    allowed = modality_mask(modality, expert_ranges, E)
    s_masked = np.where(allowed, s, -np.inf)
    p = softmax(s_masked)
    idx = topk_select(s_masked, k) if topk_idx is None else np.asarray(topk_idx, dtype=np.int32)
    if np.any(~np.take_along_axis(allowed, idx.astype(np.int64), 1)):
        raise ValueError("a token was routed outside its modality's experts")
    gates = renormalised_gates(p, idx)
    counts, offsets, row_of, src_token = dispatch(idx, E)
    y_perm = expert_ffn(gather(x, src_token), offsets, w_gate[:E], w_up[:E], w_down[:E], widen=widen_experts)
    out = combine(y_perm, row_of, gates)
    for j in range(n_shared):
        wg, wu, wd = w_gate[E + j], w_up[E + j], w_down[E + j]
        if widen_experts is not None:
            wg, wu, wd = widen_experts(wg), widen_experts(wu), widen_experts(wd)
        out = out + swiglu_ffn(x, wg, wu, wd)
    return dict(logits=s, topk_idx=idx, gates=gates, offsets=offsets, row_of=row_of, src_token=src_token, out=out)


# ----------------------------------------------------------------------------
# head-local MultiHead MoE (36kr, section 02: the hidden representation split
# into heads, each head choosing its own experts in its own subspace, the
# head results fused again)
# ----------------------------------------------------------------------------

def forward_headlocal(x, w_router, bias, w_gate, w_up, w_down, n_heads, head_dim, k, topk_idx=None,
                      widen_experts=None):
    """Head-local MoE: x [T, n_heads*head_dim] is split into head slices
    x_j = x[:, j*head_dim:(j+1)*head_dim]; head j scores its own experts,
    s_j = x_j W_router[j]^T + b[j] ([E_h] per head), takes the softmax, the
    top-k (ties to the lowest index) and renormalised gates, runs the chosen
    head-local SwiGLU experts (head_dim -> inter -> head_dim, weights
    w_gate/w_up [H, E_h, inter, head_dim], w_down [H, E_h, head_dim, inter])
    and the head outputs are concatenated back into out [T, n_heads*head_dim].
    topk_idx [H, T, k] (optional) fixes the routing decision.
    """
    T = x.shape[0]
    out = np.zeros((T, n_heads * head_dim), dtype=np.float64)
    idx_all, gates_all, logits_all = [], [], []
    for j in range(n_heads):
        cols = slice(j * head_dim, (j + 1) * head_dim)
        xj = x[:, cols]
        wr = w_router[j] if widen_experts is None else widen_experts(w_router[j])
        s = xj @ wr.T
        if bias is not None:
            s = s + np.asarray(bias[j], dtype=np.float64)[None, :]
        p = softmax(s)
        idx = topk_select(s, k) if topk_idx is None else np.asarray(topk_idx[j], dtype=np.int32)
        gates = renormalised_gates(p, idx)
        E_h = wr.shape[0]
        _, offsets, row_of, src_token = dispatch(idx, E_h)
        y_perm = expert_ffn(gather(xj, src_token), offsets, w_gate[j], w_up[j], w_down[j], widen=widen_experts)
        out[:, cols] = combine(y_perm, row_of, gates)
        idx_all.append(idx)
        gates_all.append(gates)
        logits_all.append(s)
    return dict(out=out, topk_idx=np.stack(idx_all), gates=np.stack(gates_all), logits=np.stack(logits_all))


def forward_bits(inp: dict, tokens=None, topk_idx=None):
    """Convenience: run ``forward`` on the bf16-bit input dict of moe_inputs.

    ``tokens`` selects a subset of token rows (the layer is per-token, so the
    output rows of a subset equal the same rows of the full batch).  Expert
    weights are widened per expert to bound memory.
    """
    cfg = inp["cfg"]
    xb = inp["x"] if tokens is None else inp["x"][np.asarray(tokens)]
    if cfg.head_local:
        return forward_headlocal(widen_bf16(xb), inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                                 inp["w_down"], cfg.n_heads, cfg.head_dim, cfg.top_k, topk_idx=topk_idx,
                                 widen_experts=widen_bf16)
    if cfg.n_shared or cfg.modality_experts:
        mod = inp["modality"] if tokens is None else inp["modality"][np.asarray(tokens)]
        return forward_ext(widen_bf16(xb), widen_bf16(inp["w_lat"]), widen_bf16(inp["w_head"]), inp["bias"],
                           inp["w_gate"], inp["w_up"], inp["w_down"], cfg.n_heads, cfg.head_dim, cfg.top_k,
                           modality=mod, expert_ranges=cfg.modality_experts, n_shared=cfg.n_shared,
                           topk_idx=topk_idx, widen_experts=widen_bf16)
    return forward(widen_bf16(xb), widen_bf16(inp["w_lat"]), widen_bf16(inp["w_head"]),
                   inp["bias"], inp["w_gate"], inp["w_up"], inp["w_down"],
                   cfg.n_heads, cfg.head_dim, cfg.top_k, topk_idx=topk_idx,
                   widen_experts=widen_bf16)
