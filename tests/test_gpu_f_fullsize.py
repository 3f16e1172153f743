"""The three large workloads at full size, in the launch configuration the
benchmark times: routing and outputs on sampled tokens against the oracle,
the whole permutation bit-exact, and moe_forward == the staged calls."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n_sample", [("chunk", 256), ("clip", 256), ("refiner", 256)])
def test_full_size_workload(name, n_sample):
    inp = mi.make_inputs(name)
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, gate, logits = dev.route()
    offsets, row_of, src, x_perm = dev.dispatch(idx)
    act, y = dev.ffn(x_perm, offsets)
    out = dev.combine(y, row_of, gate)
    assert dev.status() == 0
    idx_np = idx.cpu().numpy()
    # permutation: all T*k pairs, bit-exact against the oracle's counting sort
    G.check_dispatch(idx_np, cfg.E, offsets.cpu().numpy(), row_of.cpu().numpy(), src.cpu().numpy())
    counts = np.diff(offsets.cpu().numpy())
    assert counts.sum() == cfg.T * cfg.top_k
    # sampled tokens: logits, routing, gates, output rows
    tok = mi.sample_tokens(cfg.T, n_sample, seed=5)
    s_ref = G.oracle_logits(inp, tok)
    G.check_routing(s_ref, idx_np[tok], gate.cpu().numpy()[tok], cfg.top_k, logits[tok].cpu().numpy())
    src_np = src.cpu().numpy()
    rows = np.random.default_rng(1).choice(cfg.T * cfg.top_k, 64, replace=False)
    np.testing.assert_array_equal(G.bits(x_perm[torch.from_numpy(rows).cuda()]), inp["x"][src_np[rows]])
    ref = O.forward_bits(inp, tokens=tok, topk_idx=idx_np[tok])
    G.check_out(G.host_f64(out[torch.from_numpy(tok).cuda()]), ref["out"])
    out2 = dev.forward()
    assert dev.status() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    if name == "clip":   # the skew the workload asks for
        assert counts.max() >= 0.9 * cfg.T and counts.min() > 0


@pytest.mark.parametrize("fuse", [1, 2, 3])
def test_full_clip_fused_forward_sampled(fuse):
    # moe_forward_fused at the clip size, each fusion choice: sampled tokens
    # against the oracle; with the gather fused alone, the bits of moe_forward
    inp = mi.make_inputs("clip")
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, _, _ = dev.route(want_logits=False)
    out = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward_fused(dev.dims, dev.x, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, out, fuse, dev.ws)
    assert dev.status() == 0
    tok = mi.sample_tokens(cfg.T, 128, seed=23 + fuse)
    ref = O.forward_bits(inp, tokens=tok, topk_idx=idx.cpu().numpy()[tok])
    G.check_out(G.host_f64(out[torch.from_numpy(tok).cuda()]), ref["out"])
    if fuse == 1:
        assert torch.equal(out.view(torch.int16), dev.forward().view(torch.int16))
