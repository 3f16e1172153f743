"""Folded router (W_eff = W_head W_lat prepared once, one hi/lo GEMM) vs the
oracle: same logits bar, routing, gates and layer output as the two-stage
router."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _w_router(dev):
    cfg = dev.cfg
    w = torch.empty((cfg.E, 2 * cfg.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_router(dev.dims, dev.w_lat, dev.w_head, w)
    return w


def test_prepared_router_weights_match_the_product():
    inp = G.small_inputs(T=8, d=512, E=40, inter=64)
    dev = G.Dev(inp)
    w = G.host_f64(_w_router(dev))
    d = inp["cfg"].d
    ref = O.widen_bf16(inp["w_head"]) @ O.widen_bf16(inp["w_lat"])
    hi, lo = w[:, :d], w[:, d:]
    err = np.abs(hi + lo - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err
    # hi is the bf16 rounding of W_eff: |W_eff - hi| <= half a bf16 ulp of W_eff (plus fp32 sum error)
    assert np.all(np.abs(ref - hi) <= np.abs(ref) * 2.0 ** -8 + 1e-7)


@pytest.mark.parametrize("kw", [
    dict(T=256, d=512, E=16, inter=128),
    dict(T=129, d=1024, E=64, inter=64, router_init="uniform"),
    dict(T=300, d=256, E=256, inter=64, top_k=8),
    dict(T=333, d=768, E=40, inter=64, top_k=1),
])
def test_folded_router_matches_oracle(kw):
    inp = G.small_inputs(**kw)
    dev = G.Dev(inp)
    cfg = inp["cfg"]
    w = _w_router(dev)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_route_folded(dev.dims, dev.x, w, dev.bias, idx, gate, logits, dev.ws)
    assert dev.status() == 0
    G.check_routing(G.oracle_logits(inp), idx.cpu().numpy(), gate.cpu().numpy(), cfg.top_k, logits.cpu().numpy())


@pytest.mark.parametrize("name", ["tiny", "frame"])
def test_folded_forward_matches_oracle(name):
    inp = mi.make_inputs(name)
    dev = G.Dev(inp)
    cfg = inp["cfg"]
    w = _w_router(dev)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward_folded(dev.dims, dev.x, w, dev.bias, dev.w13, dev.w_down, out, dev.ws)
    assert dev.status() == 0
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    moe.moe_route_folded(dev.dims, dev.x, w, dev.bias, idx, gate, None, dev.ws)
    idx_np = idx.cpu().numpy()
    G.check_routing(G.oracle_logits(inp), idx_np, gate.cpu().numpy(), cfg.top_k)
    ref = O.forward_bits(inp, topk_idx=idx_np)
    G.check_out(G.host_f64(out), ref["out"])


def test_folded_router_full_clip_sampled():
    inp = mi.make_inputs("clip")
    dev = G.Dev(inp)
    cfg = inp["cfg"]
    w = _w_router(dev)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_route_folded(dev.dims, dev.x, w, dev.bias, idx, gate, logits, dev.ws)
    assert dev.status() == 0
    tok = mi.sample_tokens(cfg.T, 512, seed=11)
    G.check_routing(G.oracle_logits(inp, tok), idx.cpu().numpy()[tok], gate.cpu().numpy()[tok], cfg.top_k,
                    logits[torch.from_numpy(tok).cuda()].cpu().numpy())
