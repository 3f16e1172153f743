"""Whole layer on the GPU (stages and moe_forward) vs the oracle."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _full_check(inp):
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, gate, logits = dev.route()
    offsets, row_of, src, x_perm = dev.dispatch(idx)
    act, y = dev.ffn(x_perm, offsets)
    out = dev.combine(y, row_of, gate)
    assert dev.status() == 0
    idx_np = idx.cpu().numpy()
    G.check_routing(G.oracle_logits(inp), idx_np, gate.cpu().numpy(), cfg.top_k, logits.cpu().numpy())
    G.check_dispatch(idx_np, cfg.E, offsets.cpu().numpy(), row_of.cpu().numpy(), src.cpu().numpy())
    np.testing.assert_array_equal(G.bits(x_perm), inp["x"][src.cpu().numpy()])
    ref = O.forward_bits(inp, topk_idx=idx_np)
    stats = G.check_out(G.host_f64(out), ref["out"])
    # moe_forward runs the same kernels: identical bits
    out2 = dev.forward()
    assert dev.status() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    return stats


def test_tiny_workload():
    _full_check(mi.make_inputs("tiny"))


def test_frame_workload():
    _full_check(mi.make_inputs("frame"))


@pytest.mark.parametrize("kw", [
    dict(T=1, d=512, E=16, inter=128),
    dict(T=129, d=512, E=16, inter=128),
    dict(T=2049, d=256, E=256, inter=64, top_k=8),
    dict(T=600, d=320, E=20, inter=192, top_k=1),
    dict(T=300, d=512, E=6, inter=128, top_k=6),
])
def test_edge_shapes(kw):
    _full_check(G.small_inputs(**kw))


def test_all_tokens_on_six_experts():
    inp = G.small_inputs(T=1000, d=512, E=64, inter=128)
    b = np.zeros(64, np.float32)
    b[[1, 2, 40, 41, 62, 63]] = 80.0
    inp["bias"] = b
    _full_check(inp)


def test_forward_is_deterministic():
    inp = mi.make_inputs("tiny")
    dev = G.Dev(inp)
    a = dev.forward()
    b = dev.forward()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_host_buffers():
    inp = mi.make_inputs("tiny")
    dev = G.Dev(inp)
    ref = dev.forward()
    ws = moe.alloc_workspace(moe.moe_workspace_size_host(dev.dims))
    xh = dev.x.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    moe.moe_forward_host(dev.dims, xh, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, oh, ws)
    assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("T,pinned,heads", [(8193, True, 12), (20000, True, 12), (9000, False, 12), (20000, True, 1)])
def test_forward_host_chunks_match_one_forward(T, pinned, heads):
    # 2 or 3 token chunks with a ragged last one, copies overlapping compute
    # (pinned) or serialised with it (pageable): the same bits as one
    # moe_forward over the whole batch, and the oracle on tokens of every
    # chunk.  With one 256-dim head the whole batch routes on chip, so it
    # runs as one piece.
    inp = G.small_inputs(T=T, d=512, E=32, inter=128, seed=3, n_heads=heads, head_dim=256)
    dev = G.Dev(inp)
    ref = dev.forward()
    idx, _, _ = dev.route(want_logits=False)
    assert dev.status() == 0
    ws = moe.alloc_workspace(moe.moe_workspace_size_host(dev.dims))
    xh = dev.x.cpu()
    oh = torch.full_like(xh, float("nan"))
    if pinned:
        xh, oh = xh.pin_memory(), oh.pin_memory()
    moe.moe_forward_host(dev.dims, xh, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, oh, ws)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))
    rng = np.random.default_rng(T)
    tok = np.unique(np.r_[0, T - 1, T // 2, rng.choice(T, 120, replace=False)])
    want = O.forward_bits(inp, tokens=tok, topk_idx=idx.cpu().numpy()[tok])
    G.check_out(G.host_f64(oh[tok]), want["out"])


@pytest.mark.parametrize("kw", [dict(T=3000, d=512, E=32, inter=256), dict(T=77, d=4096, E=8, inter=1024),
                                dict(T=1, d=512, E=16, inter=128),
                                dict(T=500, d=256, E=8, inter=192)])   # 2*inter = 384: 128-wide N tiles
def test_gathered_gemm1_equals_gemm1_on_x_perm(kw):
    inp = G.small_inputs(**kw)
    dev = G.Dev(inp)
    cfg = inp["cfg"]
    idx, gate, _ = dev.route(want_logits=False)
    offsets, row_of, src, x_perm = dev.dispatch(idx)
    act_ref, _ = dev.ffn(x_perm, offsets)
    off2 = torch.empty_like(offsets)
    row2 = torch.empty_like(row_of)
    src2 = torch.empty_like(src)
    moe.moe_dispatch_indices(dev.dims, idx, off2, row2, src2, dev.ws)
    assert torch.equal(off2, offsets) and torch.equal(row2, row_of) and torch.equal(src2, src)
    act = torch.full_like(act_ref, float("nan"))
    moe.moe_expert_gemm1_gather(dev.dims, dev.x, src, offsets, dev.w13, act, dev.ws)
    assert dev.status() == 0
    assert torch.equal(act.view(torch.int16), act_ref.view(torch.int16))


def test_pipeline_wait_timeout_is_reported_and_the_context_survives():
    # the loader issues nothing: the kernel's waits run out after 20 ms
    ws = moe.alloc_workspace(1 << 20)
    moe.moe_clear_device_status(ws)
    moe.moe_selftest_timeout(ws, 20_000)
    assert moe.moe_get_device_status(ws) & moe.binding.MOE_DEV_TIMEOUT
    # the GPU still computes correctly afterwards (tensor memory was released)
    inp = mi.make_inputs("tiny")
    dev = G.Dev(inp)
    idx, gate, _ = dev.route(want_logits=False)
    out = dev.forward()
    assert dev.status() == 0
    ref = O.forward_bits(inp, topk_idx=idx.cpu().numpy())
    G.check_out(G.host_f64(out), ref["out"])


def test_forward_captured_in_a_cuda_graph_replays_with_new_inputs():
    # group sizes stay on the device, so one captured moe_forward serves any
    # routing: replaying it on new x gives the bits of a direct call
    inp = G.small_inputs(T=3000, d=512, E=32, inter=256, seed=5)
    dev = G.Dev(inp)
    ref1 = dev.forward()  # first launches (and kernel attributes) outside the capture
    g2 = torch.Generator(device="cpu").manual_seed(11)
    x2 = (torch.randn(dev.x.shape, generator=g2) * 1.5).to(torch.bfloat16).cuda()
    x_buf = dev.x.clone()
    ref2 = torch.empty_like(ref1)
    moe.moe_forward(dev.dims, x2, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, ref2, dev.ws)
    torch.cuda.synchronize()
    out = torch.full_like(ref1, float("nan"))
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        moe.moe_forward(dev.dims, x_buf, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, out, dev.ws)
    graph.replay()
    torch.cuda.synchronize()
    assert dev.status() == 0
    assert torch.equal(out.view(torch.int16), ref1.view(torch.int16))
    x_buf.copy_(x2)
    graph.replay()
    torch.cuda.synchronize()
    assert dev.status() == 0
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))
    assert not torch.equal(ref1.view(torch.int16), ref2.view(torch.int16))


@pytest.mark.parametrize("router,fuse", [("latent", 0), ("folded", 0), ("latent", 1), ("latent", 3)])
def test_layer_wrapper_runs_the_entry_point_it_names(router, fuse):
    # MoeLayer(router=, fuse=) is plumbing only: its output has the bits of
    # the entry point it selects (each of those is checked against the oracle
    # in its own tests)
    inp = mi.make_inputs("tiny")
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    layer = moe.MoeLayer(dev.dims, dev.w_lat, dev.w_head, dev.bias, G.dev_bf16(inp["w_gate"]),
                         G.dev_bf16(inp["w_up"]), dev.w_down, router=router, fuse=fuse)
    got = layer.forward(dev.x)
    assert layer.device_status() == 0
    want = torch.empty_like(got)
    if router == "folded":
        w = torch.empty((cfg.E, 2 * cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_prepare_router(dev.dims, dev.w_lat, dev.w_head, w)
        moe.moe_forward_folded(dev.dims, dev.x, w, dev.bias, dev.w13, dev.w_down, want, dev.ws)
    else:
        moe.moe_forward_fused(dev.dims, dev.x, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, want, fuse,
                              dev.ws)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_tiny_forward_matches_the_stored_oracle_sample():
    # the stored fp64 oracle sample (tests/golden/tiny_oracle.json, written
    # by oracle/ only): same routing on every sampled token (all clear of
    # near-ties) and the sampled outputs within the layer's bars
    import json
    import pathlib
    g = json.loads((pathlib.Path(__file__).resolve().parent / "golden" / "tiny_oracle.json").read_text())
    inp = mi.make_inputs("tiny")
    dev = G.Dev(inp)
    idx, _, _ = dev.route(want_logits=False)
    out = G.host_f64(dev.forward())
    assert dev.status() == 0
    t = g["tokens"]
    assert min(g["topk_gap"]) > 2e-3
    np.testing.assert_array_equal(idx.cpu().numpy()[t], np.array(g["topk_idx"]))
    G.check_out(out[t, :g["out_cols"]], np.array(g["out"]))
