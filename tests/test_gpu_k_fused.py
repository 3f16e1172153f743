"""Fused steps of the layer (the 36kr article, section 02: the operator
library fuses calculation steps to cut intermediates and memory traffic)
against the fp64 oracle:

* expert GEMM-1 with the sorting gather in its operand loads
  (moe_expert_gemm1_gather), element-wise;
* expert GEMM-2 with the gate in its epilogue (moe_expert_gemm2_gated) and
  the unweighted row combine (moe_combine_rows);
* moe_forward_fused with every choice of fusions, end to end;
* a gathered row whose source index is outside x: read as zeros, flagged;
* the SwiGLU epilogue's silu over the whole range it meets, element-wise,
  on inputs whose GEMM sums are exact in fp32.
"""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from fine_grained_moe_02_b300 import binding as B
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

FUSIONS = [0, B.MOE_FUSE_GATHER, B.MOE_FUSE_GATE, B.MOE_FUSE_GATHER | B.MOE_FUSE_GATE]


def _oracle_act(xw, offsets, wg, wu):
    """silu(x W_gate^T) * (x W_up^T) per expert group, fp64 (also returns g, u)."""
    E = len(offsets) - 1
    R = xw.shape[0]
    g = np.zeros((R, wg.shape[1]))
    u = np.zeros_like(g)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            g[lo:hi] = xw[lo:hi] @ O.widen_bf16(wg[e]).T
            u[lo:hi] = xw[lo:hi] @ O.widen_bf16(wu[e]).T
    return O.silu(g) * u, g, u


def _gathered_case(T, d, E, I, counts, seed, exact=False):
    """x [T, d], src_token [R] (rows drawn from the tokens), group offsets and
    expert weights.  exact=True: small integers for x and multiples of 1/8 for
    sparse weights, so every GEMM sum is exact in fp32 whatever its order."""
    g = np.random.default_rng(seed)
    R = int(sum(counts))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    src = g.integers(0, T, size=R).astype(np.int32)
    if exact:
        x = g.integers(-2, 3, size=(T, d)).astype(np.float32)
        def w(shape):
            k = g.integers(-16, 17, size=shape).astype(np.float32) / 8.0
            return k * (g.random(shape) < 1.0 / 16)
        wg, wu = w((E, I, d)), w((E, I, d))
    else:
        x = g.standard_normal((T, d)).astype(np.float32)
        wg = (g.standard_normal((E, I, d)) / np.sqrt(d)).astype(np.float32)
        wu = (g.standard_normal((E, I, d)) / np.sqrt(d)).astype(np.float32)
    return (R, offsets, src, mi.f32_to_bf16_bits(x), mi.f32_to_bf16_bits(wg), mi.f32_to_bf16_bits(wu))


def _run_gemm1(T, d, E, I, offsets, src, x, wg, wu, gathered, status=0):
    """act of the R = offsets[-1] rows.  dims.T covers both x's T tokens and
    the R rows (top_k = 1): x is [dims.T, d] and src_token indexes it."""
    R = int(offsets[-1])
    Td = max(T, R, 1)
    dims = moe.moe_dims.make(Td, d, E, I, 1, n_heads=1, head_dim=256)
    ws = moe.alloc_workspace(moe.moe_scratch_size(dims))
    w13 = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_weights(dims, G.dev_bf16(wg), G.dev_bf16(wu), w13)
    act = torch.full((Td, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    off_d = torch.from_numpy(offsets).cuda()
    if gathered:
        xbuf = np.zeros((Td, d), np.uint16)
        xbuf[:T] = x
        src_d = torch.from_numpy(np.r_[src, np.zeros(Td - R, np.int32)].astype(np.int32)).cuda()
        moe.moe_expert_gemm1_gather(dims, G.dev_bf16(xbuf), src_d, off_d, w13, act, ws)
    else:
        xp = np.zeros((Td, d), np.uint16)
        xp[:R] = x[src]
        moe.moe_expert_gemm1(dims, G.dev_bf16(xp), off_d, w13, act, ws)
    assert moe.moe_get_device_status(ws) == status
    return G.host_f64(act)[:R]


@pytest.mark.parametrize("gathered", [False, True])
def test_silu_is_accurate_over_the_whole_range_elementwise(gathered):
    # g and u exact in fp32 (integer-valued x, sparse multiples of 1/8 as
    # weights), g spread over about [-20, 20]: the only errors left are silu
    # itself and act's one bf16 rounding (2^-9 relative), so every element
    # must be within 2^-8 of the oracle relative to its own size -- including
    # g in [-12, -3], where 1 + tanh(g/2) would cancel.
    T, d, E, I = 700, 256, 3, 128
    counts = [300, 0, 211]
    R, offsets, src, x, wg, wu = _gathered_case(T, d, E, I, counts, seed=21, exact=True)
    act = _run_gemm1(T, d, E, I, offsets, src, x, wg, wu, gathered)
    ref, g, u = _oracle_act(O.widen_bf16(x[src]), offsets, wg, wu)
    assert np.all(np.abs(g) < 2 ** 20) and np.all(g * 8 == np.round(g * 8))   # exact-sum inputs
    neg = (g > -12) & (g < -3) & (u != 0)
    assert neg.sum() > 2000 and (g < -14).any() and (g > 14).any()            # the range is covered
    err = np.abs(act - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref)), float((err / np.maximum(np.abs(ref), 1e-300)).max())


@pytest.mark.parametrize("T,d,E,I,counts", [
    (200, 128, 1, 128, [128]),                       # one full tile
    (300, 256, 2, 128, [200, 77]),                   # ragged tails
    (500, 512, 4, 256, [0, 300, 0, 129]),            # empty groups
    (400, 320, 3, 192, [1, 64, 130]),                # 2*inter = 384: 128-wide N tiles
    (900, 4096, 3, 1024, [260, 5, 128]),             # production widths
    (2000, 1024, 8, 512, [17, 0, 400, 1, 128, 255, 3, 90]),
])
def test_gathered_gemm1_matches_oracle(T, d, E, I, counts):
    # act[r] = silu(x[src[r]] W_gate^T) * (x[src[r]] W_up^T), rows fetched from x by src_token
    R, offsets, src, x, wg, wu = _gathered_case(T, d, E, I, counts, seed=7)
    act = _run_gemm1(T, d, E, I, offsets, src, x, wg, wu, gathered=True)
    ref, _, _ = _oracle_act(O.widen_bf16(O.gather(x, src)), offsets, wg, wu)
    assert np.isfinite(act).all()
    rel = np.linalg.norm(act - ref) / np.linalg.norm(ref)
    assert rel <= 5e-3, rel
    assert np.abs(act - ref).max() <= G.OUT_MAX_ABS
    # and the same bits as GEMM-1 on the gathered x_perm
    np.testing.assert_array_equal(act, _run_gemm1(T, d, E, I, offsets, src, x, wg, wu, gathered=False))


def test_gathered_gemm1_reads_a_source_row_outside_x_as_zeros():
    # a src_token entry outside [0, T) is never dereferenced: the row reads
    # as zeros (act 0) and MOE_DEV_BAD_SOURCE_ROW is set; every other row is
    # untouched
    T, d, E, I = 300, 256, 2, 128
    R, offsets, src, x, wg, wu = _gathered_case(T, d, E, I, [200, 77], seed=5)
    good = _run_gemm1(T, d, E, I, offsets, src, x, wg, wu, gathered=True)
    bad_src = src.copy()
    bad_src[[5, 150, 276]] = [T + 1000, -3, 2 ** 31 - 1]
    act = _run_gemm1(T, d, E, I, offsets, bad_src, x, wg, wu, gathered=True, status=B.MOE_DEV_BAD_SOURCE_ROW)
    assert np.all(act[[5, 150, 276]] == 0)
    keep = np.ones(R, bool)
    keep[[5, 150, 276]] = False
    np.testing.assert_array_equal(act[keep], good[keep])


def test_gated_gemm2_and_row_combine_match_oracle():
    inp = G.small_inputs(T=3000, d=512, E=32, inter=256, seed=9)
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, gate, _ = dev.route(want_logits=False)
    offsets, row_of, src, x_perm = dev.dispatch(idx)
    act, y = dev.ffn(x_perm, offsets)
    yg = torch.full_like(y, float("nan"))
    moe.moe_expert_gemm2_gated(dev.dims, act, offsets, dev.w_down, src, row_of, gate, yg, dev.ws)
    out = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_rows(dev.dims, yg, row_of, out)
    assert dev.status() == 0
    # y rows scaled by their own gate: against the oracle's expert outputs times the gate
    src_np, row_np, gate_np = src.cpu().numpy(), row_of.cpu().numpy(), gate.cpu().numpy().astype(np.float64)
    g_row = np.zeros(cfg.T * cfg.top_k)
    g_row[row_np.reshape(-1)] = gate_np.reshape(-1)
    y_ref = O.expert_ffn(O.widen_bf16(inp["x"][src_np]), offsets.cpu().numpy(), inp["w_gate"], inp["w_up"],
                         inp["w_down"], widen=O.widen_bf16)
    G.check_out(G.host_f64(yg), g_row[:, None] * y_ref)
    ref = O.forward_bits(inp, topk_idx=idx.cpu().numpy())
    G.check_out(G.host_f64(out), ref["out"])


def _fused_check(inp, fuse):
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, _, _ = dev.route(want_logits=False)
    out = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward_fused(dev.dims, dev.x, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, out, fuse, dev.ws)
    assert dev.status() == 0
    ref = O.forward_bits(inp, topk_idx=idx.cpu().numpy())
    stats = G.check_out(G.host_f64(out), ref["out"])
    if not fuse & B.MOE_FUSE_GATE:   # the gather fusion alone changes no bit
        assert torch.equal(out.view(torch.int16), dev.forward().view(torch.int16))
    return stats


@pytest.mark.parametrize("fuse", FUSIONS)
@pytest.mark.parametrize("name", ["tiny", "frame"])
def test_fused_forward_matches_oracle(name, fuse):
    _fused_check(mi.make_inputs(name), fuse)


@pytest.mark.parametrize("fuse", FUSIONS[1:])
@pytest.mark.parametrize("kw", [
    dict(T=1, d=512, E=16, inter=128),
    dict(T=2049, d=256, E=256, inter=64, top_k=8),
    dict(T=600, d=320, E=20, inter=192, top_k=1),
    dict(T=5000, d=512, E=64, inter=128),
])
def test_fused_forward_edge_shapes(kw, fuse):
    _fused_check(G.small_inputs(**kw), fuse)


def test_fused_forward_rejects_unknown_fusion_bits():
    inp = mi.make_inputs("tiny")
    dev = G.Dev(inp)
    out = torch.empty((inp["cfg"].T, inp["cfg"].d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_fused(dev.dims, dev.x, dev.w_lat, dev.w_head, dev.bias, dev.w13, dev.w_down, out, 4, dev.ws)
    assert e.value.code == B.MOE_ERR_INVALID_ARG
