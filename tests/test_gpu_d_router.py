"""Router (two tcgen05 GEMMs with hi/lo latent split + fused top-k) vs oracle."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kw", [
    dict(T=256, d=512, E=16, inter=128),                               # the tiny workload's router
    dict(T=1, d=512, E=16, inter=128),
    dict(T=129, d=1024, E=64, inter=64, router_init="uniform"),
    dict(T=300, d=256, E=256, inter=64, top_k=8),
    dict(T=200, d=512, E=6, inter=64, top_k=6),                         # k == E: gates = full softmax
    dict(T=333, d=768, E=40, inter=64, top_k=1),                        # E not a power of two
    dict(T=130, d=128, E=128, inter=64, n_heads=2, head_dim=128),      # other head geometry
    dict(T=200, d=256, E=32, inter=64, n_heads=4, head_dim=64),        # fused router, small heads
    dict(T=150, d=512, E=48, inter=64, n_heads=4, head_dim=192),       # fused router, 3 chunks per head
    dict(T=140, d=256, E=24, inter=64, n_heads=1, head_dim=512),       # two-stage only
    dict(T=1000, d=1024, E=128, inter=64),                              # on-chip: several head groups
])
@pytest.mark.parametrize("path", ["auto", "two_stage", "fused"])
def test_router_matches_oracle(kw, path):
    # auto = moe_route, which picks the on-chip path for small batches
    inp = G.small_inputs(**kw)
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    if path == "auto":
        idx, gate, logits = dev.route()
    elif path == "two_stage":
        idx, gate, logits = dev.route_two_stage()
    else:
        if cfg.head_dim % 64 or cfg.head_dim > 256:
            pytest.skip("the on-chip router covers head_dim % 64 == 0, <= 256")
        idx, gate, logits = dev.route_fused()
    assert dev.status() == 0
    s_ref = G.oracle_logits(inp)
    stats = G.check_routing(s_ref, idx.cpu().numpy(), gate.cpu().numpy(), cfg.top_k, logits.cpu().numpy())
    assert stats["near_ties"] <= max(3, cfg.T // 50)


def test_router_bias_forces_experts():
    inp = G.small_inputs(T=500, d=256, E=32, inter=64)
    b = np.zeros(32, np.float32)
    b[[3, 9, 12, 20, 27, 31]] = np.array([600, 500, 400, 300, 200, 100], np.float32)
    inp["bias"] = b
    dev = G.Dev(inp)
    idx, gate, logits = dev.route()
    got = idx.cpu().numpy()
    assert np.all(got == np.array([3, 9, 12, 20, 27, 31]))
    G.check_routing(G.oracle_logits(inp), got, gate.cpu().numpy(), 6, logits.cpu().numpy())


def test_router_without_logits_output_gives_same_routing():
    inp = G.small_inputs(T=700, d=512, E=64, inter=64)
    dev = G.Dev(inp)
    i1, g1, _ = dev.route(want_logits=True)
    i2, g2, _ = dev.route(want_logits=False)
    assert torch.equal(i1, i2) and torch.equal(g1, g2)


def test_fused_router_full_clip_sampled():
    inp = mi.make_inputs("clip")
    dev = G.Dev(inp)
    cfg = inp["cfg"]
    idx, gate, logits = dev.route_fused()
    assert dev.status() == 0
    tok = mi.sample_tokens(cfg.T, 512, seed=13)
    G.check_routing(G.oracle_logits(inp, tok), idx.cpu().numpy()[tok], gate.cpu().numpy()[tok], cfg.top_k,
                    logits[torch.from_numpy(tok).cuda()].cpu().numpy())


@pytest.mark.parametrize("path", ["two_stage", "fused", "folded"])
def test_exact_ties_go_to_the_lower_index(path):
    # experts e, e+8, e+16, e+24 share a W_head row and a bias, so they score
    # exactly alike on every token: the top-6 boundary falls inside a tie
    # group, where only the lower expert indices may be taken, in index order
    inp = G.small_inputs(T=400, d=512, E=32, inter=64, seed=9)
    cfg = inp["cfg"]
    ng, E = 8, 32
    inp["w_head"] = np.ascontiguousarray(inp["w_head"][np.arange(E) % ng])
    gb = np.random.default_rng(4).normal(0.0, 2.0, ng).astype(np.float32)
    inp["bias"] = np.ascontiguousarray(gb[np.arange(E) % ng])
    dev = G.Dev(inp)
    if path == "two_stage":
        idx, gate, logits = dev.route_two_stage()
    elif path == "fused":
        idx, gate, logits = dev.route_fused()
    else:
        w = torch.empty((E, 2 * cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_prepare_router(dev.dims, dev.w_lat, dev.w_head, w)
        idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
        gate = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
        logits = torch.empty((cfg.T, E), dtype=torch.float32, device="cuda")
        moe.moe_route_folded(dev.dims, dev.x, w, dev.bias, idx, gate, logits, dev.ws)
    assert dev.status() == 0
    lg = logits.cpu().numpy()
    members = [np.arange(g, E, ng) for g in range(ng)]
    for g in range(ng):
        assert np.all(lg[:, members[g]] == lg[:, [g]])  # tied experts: bit-identical logits
    gv = G.oracle_logits(inp)[:, :ng]  # one value per tie group
    order = np.argsort(-gv, axis=1, kind="stable")
    want = np.array([np.concatenate([members[g] for g in row])[:cfg.top_k] for row in order])
    clear = np.min(np.diff(np.sort(gv, axis=1), axis=1), axis=1) > 1e-3  # groups apart by > 1e-3
    assert clear.sum() > 0.9 * cfg.T
    np.testing.assert_array_equal(idx.cpu().numpy()[clear], want[clear])
    g = gate.cpu().numpy()[clear]
    same = np.take_along_axis(lg[clear], idx.cpu().numpy()[clear], axis=1)
    # equal logits get equal gates
    for t in range(g.shape[0]):
        for a in range(cfg.top_k):
            for b in range(a + 1, cfg.top_k):
                if same[t, a] == same[t, b]:
                    assert g[t, a] == g[t, b]
