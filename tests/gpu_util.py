"""Helpers for the GPU parity tests: upload seeded inputs, run the C-ABI
stages, and compare against the fp64 oracle with the layer's parity bars.

Parity bars (fixed by the layer's specification):
  * router logits: max-abs error <= 1e-3
  * expert indices and the permutation: the chosen set bit-exact wherever the
    oracle's k-th to (k+1)-th logit margin exceeds 1e-3, the slot order
    bit-exact where adjacent in-set gaps also exceed 2e-3 (otherwise a valid
    descending order); on near-tie tokens the GPU's set must be a valid top-k
    (each chosen logit >= oracle k-th logit - 2e-3); the permutation
    bit-exact against the oracle's counting sort of the GPU's ids
  * layer output: relative Frobenius error <= 1e-2 and max-abs <= 5e-2
  * gates: max-abs <= 1e-3 (diagnostic), sum to 1 within 1e-6
"""
from __future__ import annotations

import numpy as np
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O

LOGIT_TOL = 1e-3
MARGIN = 1e-3
OUT_REL_FRO = 1e-2
OUT_MAX_ABS = 5e-2
GATE_TOL = 1e-3


def dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dims_of(cfg) -> moe.moe_dims:
    return moe.moe_dims.make(cfg.T, cfg.d, cfg.E, cfg.inter, cfg.top_k, cfg.n_heads, cfg.head_dim)


class Dev:
    """Device copies of one workload's inputs, plus w13 and a workspace."""

    def __init__(self, inp: dict):
        self.inp = inp
        cfg = self.cfg = inp["cfg"]
        self.dims = dims_of(cfg)
        self.x = dev_bf16(inp["x"])
        self.w_lat = dev_bf16(inp["w_lat"])
        self.w_head = dev_bf16(inp["w_head"])
        self.bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).cuda()
        self.w_down = dev_bf16(inp["w_down"])
        wg, wu = dev_bf16(inp["w_gate"]), dev_bf16(inp["w_up"])
        n_exp = wg.shape[0]                      # routed + shared experts
        self.w13 = torch.empty((n_exp, 2 * cfg.inter, cfg.d), dtype=torch.bfloat16, device="cuda")
        dims_w = moe.moe_dims.make(cfg.T, cfg.d, n_exp, cfg.inter, min(cfg.top_k, n_exp), cfg.n_heads, cfg.head_dim)
        moe.moe_prepare_weights(dims_w, wg, wu, self.w13)
        del wg, wu
        self.modality = torch.from_numpy(inp["modality"]).cuda() if "modality" in inp else None
        self.ext = moe.moe_ext.make(cfg.n_shared, cfg.modality_experts,
                                    self.modality if cfg.modality_experts else None)
        self.ws = moe.alloc_workspace(max(moe.moe_workspace_size(self.dims),
                                          moe.moe_workspace_size_ext(self.dims, self.ext)))

    # -- stages
    def route(self, want_logits=True):
        T, k, E = self.cfg.T, self.cfg.top_k, self.cfg.E
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda") if want_logits else None
        moe.moe_route(self.dims, self.x, self.w_lat, self.w_head, self.bias, idx, gate, logits, self.ws)
        return idx, gate, logits

    def route_two_stage(self):
        T, k, E = self.cfg.T, self.cfg.top_k, self.cfg.E
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route_two_stage(self.dims, self.x, self.w_lat, self.w_head, self.bias, idx, gate, logits, self.ws)
        return idx, gate, logits

    def route_fused(self):
        T, k, E = self.cfg.T, self.cfg.top_k, self.cfg.E
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route_fused(self.dims, self.x, self.w_lat, self.w_head, self.bias, idx, gate, logits, self.ws)
        return idx, gate, logits

    def dispatch(self, idx):
        T, k, E, d = self.cfg.T, self.cfg.top_k, self.cfg.E, self.cfg.d
        offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        row_of = torch.empty((T, k), dtype=torch.int32, device="cuda")
        src = torch.empty(T * k, dtype=torch.int32, device="cuda")
        x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device="cuda")
        moe.moe_dispatch(self.dims, self.x, idx, offsets, row_of, src, x_perm, self.ws)
        return offsets, row_of, src, x_perm

    def ffn(self, x_perm, offsets):
        rows = x_perm.shape[0]
        act = torch.empty((rows, self.cfg.inter), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((rows, self.cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_expert_ffn(self.dims, x_perm, offsets, self.w13, self.w_down, act, y, self.ws)
        return act, y

    def combine(self, y, row_of, gate):
        out = torch.empty((self.cfg.T, self.cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine(self.dims, y, row_of, gate, out)
        return out

    def forward(self):
        out = torch.empty((self.cfg.T, self.cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_forward(self.dims, self.x, self.w_lat, self.w_head, self.bias, self.w13, self.w_down, out, self.ws)
        return out

    def forward_ext(self):
        out = torch.empty((self.cfg.T, self.cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_forward_ext(self.dims, self.ext, self.x, self.w_lat, self.w_head, self.bias, self.w13, self.w_down,
                            out, self.ws)
        return out

    def route_ext(self):
        T, k, E = self.cfg.T, self.cfg.top_k, self.cfg.E
        ko = k + self.cfg.n_shared
        idx = torch.empty((T, ko), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, ko), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route_ext(self.dims, self.ext, self.x, self.w_lat, self.w_head, self.bias, idx, gate, logits,
                          self.ws)
        return idx, gate, logits

    def status(self) -> int:
        return moe.moe_get_device_status(self.ws)


# -- parity checks -----------------------------------------------------------

def oracle_logits(inp, tokens=None) -> np.ndarray:
    cfg = inp["cfg"]
    xb = inp["x"] if tokens is None else inp["x"][tokens]
    h = O.latent_projection(O.widen_bf16(xb), O.widen_bf16(inp["w_lat"]))
    return O.head_scores(h, O.widen_bf16(inp["w_head"]), inp["bias"], cfg.n_heads, cfg.head_dim)


def check_routing(s_ref: np.ndarray, idx_gpu: np.ndarray, gate_gpu: np.ndarray, k: int,
                  logits_gpu: np.ndarray | None = None) -> dict:
    """Router parity on a set of tokens; returns stats."""
    T, E = s_ref.shape
    if logits_gpu is not None:
        err = np.abs(logits_gpu.astype(np.float64) - s_ref).max()
        assert err <= LOGIT_TOL, f"logit max-abs {err}"
    idx_ref = O.topk_select(O.softmax(s_ref), k)
    srt = np.sort(s_ref, axis=1)[:, ::-1]
    margin = srt[:, k - 1] - srt[:, k] if k < E else np.full(T, np.inf)
    clear = margin > MARGIN
    # the chosen set is unique where the k-th/(k+1)-th margin exceeds the bar
    np.testing.assert_array_equal(np.sort(idx_gpu[clear], 1), np.sort(idx_ref[clear], 1))
    # slot order: unique where every adjacent gap inside the top-k exceeds two
    # logit tolerances; elsewhere it must be a valid descending order
    gaps = -np.diff(srt[:, :k], axis=1) if k > 1 else np.full((T, 1), np.inf)
    ordered = clear & np.all(gaps > 2 * LOGIT_TOL, axis=1)
    np.testing.assert_array_equal(idx_gpu[ordered], idx_ref[ordered])
    along = np.take_along_axis(s_ref, np.clip(idx_gpu, 0, E - 1).astype(np.int64), 1)
    assert np.all(np.diff(along, axis=1) <= 2 * LOGIT_TOL)
    # near ties: a valid top-k with distinct in-range ids
    assert np.all((idx_gpu >= 0) & (idx_gpu < E))
    for t in np.nonzero(~clear)[0]:
        assert len(set(idx_gpu[t].tolist())) == k
        assert np.all(s_ref[t, idx_gpu[t]] >= srt[t, k - 1] - 2 * LOGIT_TOL), (t, s_ref[t, idx_gpu[t]], srt[t, :k + 1])
    gate_ref = O.renormalised_gates(O.softmax(s_ref), idx_gpu)
    gerr = np.abs(gate_gpu - gate_ref).max()
    assert gerr <= GATE_TOL, f"gate max-abs {gerr}"
    assert np.all(np.abs(gate_gpu.astype(np.float64).sum(1) - 1) <= 1e-6)
    return dict(near_ties=int((~clear).sum()), gate_err=float(gerr))


def check_dispatch(idx_gpu: np.ndarray, E: int, offsets, row_of, src) -> None:
    counts, off_ref, row_ref, src_ref = O.dispatch(idx_gpu, E)
    np.testing.assert_array_equal(offsets, off_ref)
    np.testing.assert_array_equal(row_of, row_ref)
    np.testing.assert_array_equal(src, src_ref)


def check_out(out_gpu: np.ndarray, out_ref: np.ndarray) -> dict:
    diff = out_gpu - out_ref
    rel = np.linalg.norm(diff) / max(np.linalg.norm(out_ref), 1e-30)
    mx = np.abs(diff).max() if diff.size else 0.0
    assert rel <= OUT_REL_FRO, f"relative Frobenius {rel}"
    assert mx <= OUT_MAX_ABS, f"max-abs {mx}"
    return dict(rel_fro=float(rel), max_abs=float(mx))


def small_inputs(name="edge", seed=0, **kw):
    cfg = mi.custom_config(name, seed=seed, **kw)
    return mi.make_inputs(cfg)


def check_routing_ext(inp, s_ref, idx_gpu, gate_gpu, logits_gpu=None, tokens=None):
    """Routing parity with modality ranges and shared slots: the routed slots
    against the oracle's masked scores, then the shared slots."""
    cfg = inp["cfg"]
    k, S, E = cfg.top_k, cfg.n_shared, cfg.E
    mod = inp["modality"] if tokens is None else inp["modality"][tokens]
    allowed = O.modality_mask(mod, cfg.modality_experts, E)
    if logits_gpu is not None:
        err = np.abs(logits_gpu.astype(np.float64) - s_ref).max()
        assert err <= LOGIT_TOL, f"logit max-abs {err}"
    s_masked = np.where(allowed, s_ref, -np.inf)
    check_routing(s_masked, idx_gpu[:, :k], gate_gpu[:, :k], k)
    assert np.all(np.take_along_axis(allowed, idx_gpu[:, :k].astype(np.int64), 1))
    for j in range(S):
        assert np.all(idx_gpu[:, k + j] == E + j) and np.all(gate_gpu[:, k + j] == 1.0)
