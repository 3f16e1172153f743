"""Grouped SwiGLU expert GEMMs (tcgen05) vs the oracle, from the same x_perm."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _case(d, E, I, counts, seed=0):
    g = np.random.default_rng(seed)
    R = int(sum(counts))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = mi.f32_to_bf16_bits(g.standard_normal((R, d)).astype(np.float32))
    wg = mi.f32_to_bf16_bits((g.standard_normal((E, I, d)) / np.sqrt(d)).astype(np.float32))
    wu = mi.f32_to_bf16_bits((g.standard_normal((E, I, d)) / np.sqrt(d)).astype(np.float32))
    wd = mi.f32_to_bf16_bits((g.standard_normal((E, d, I)) / np.sqrt(I)).astype(np.float32))
    return R, offsets, x, wg, wu, wd


def _run(d, E, I, counts, seed=0):
    R, offsets, x, wg, wu, wd = _case(d, E, I, counts, seed)
    k = 1
    dims = moe.moe_dims.make(max(R, 1), d, E, I, k, n_heads=1, head_dim=256)
    ws = moe.alloc_workspace(moe.moe_scratch_size(dims))
    w13 = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_weights(dims, G.dev_bf16(wg), G.dev_bf16(wu), w13)
    xd = G.dev_bf16(x) if R else torch.zeros((1, d), dtype=torch.bfloat16, device="cuda")
    act = torch.full((max(R, 1), I), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((max(R, 1), d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(dims, xd, torch.from_numpy(offsets).cuda(), w13, G.dev_bf16(wd), act, y, ws)
    status = moe.moe_get_device_status(ws)
    return status, R, offsets, x, wg, wu, wd, G.host_f64(act)[:R], G.host_f64(y)[:R], w13


def _ref(x, offsets, wg, wu, wd):
    xw = O.widen_bf16(x)
    E = len(offsets) - 1
    act = np.zeros((xw.shape[0], wg.shape[1]))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            act[lo:hi] = O.silu(xw[lo:hi] @ O.widen_bf16(wg[e]).T) * (xw[lo:hi] @ O.widen_bf16(wu[e]).T)
    y = O.expert_ffn(xw, offsets, wg, wu, wd, widen=O.widen_bf16)
    return act, y


def test_prepare_weights_layout():
    d, E, I = 128, 3, 192
    _, _, _, wg, wu, _ = _case(d, E, I, [1, 1, 1])
    dims = moe.moe_dims.make(3, d, E, I, 1, n_heads=1, head_dim=256)
    w13 = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_weights(dims, G.dev_bf16(wg), G.dev_bf16(wu), w13)
    got = G.bits(w13)
    for e in range(E):
        for b in range(I // 64):
            np.testing.assert_array_equal(got[e, 128 * b:128 * b + 64], wg[e, 64 * b:64 * b + 64])
            np.testing.assert_array_equal(got[e, 128 * b + 64:128 * b + 128], wu[e, 64 * b:64 * b + 64])


@pytest.mark.parametrize("d,E,I,counts", [
    (128, 1, 128, [128]),                       # one full tile
    (256, 2, 128, [200, 77]),                   # ragged tails
    (512, 4, 256, [0, 300, 0, 129]),            # empty groups
    (320, 3, 192, [1, 64, 130]),                # N tiles of 128 / 64
    (4096, 3, 1024, [260, 5, 128]),             # production widths
    (1024, 8, 512, [17, 0, 400, 1, 128, 255, 3, 90]),
])
def test_expert_ffn_matches_oracle(d, E, I, counts):
    status, R, offsets, x, wg, wu, wd, act, y, _ = _run(d, E, I, counts)
    assert status == 0
    act_ref, y_ref = _ref(x, offsets, wg, wu, wd)
    assert np.isfinite(act).all() and np.isfinite(y).all()
    rel_a = np.linalg.norm(act - act_ref) / np.linalg.norm(act_ref)
    assert rel_a <= 5e-3, rel_a
    G.check_out(y, y_ref)


def test_expert_ffn_flags_bad_offsets_without_faulting():
    d, E, I = 128, 2, 64
    R, offsets, x, wg, wu, wd = _case(d, E, I, [64, 64])
    dims = moe.moe_dims.make(R, d, E, I, 1, n_heads=1, head_dim=256)
    ws = moe.alloc_workspace(moe.moe_scratch_size(dims))
    w13 = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_weights(dims, G.dev_bf16(wg), G.dev_bf16(wu), w13)
    bad = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")      # not monotone
    act = torch.zeros((R, I), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(dims, G.dev_bf16(x), bad, w13, G.dev_bf16(wd), act, y, ws)
    assert moe.moe_get_device_status(ws) & moe.binding.MOE_DEV_BAD_OFFSETS
    assert float(y.abs().max()) == 0.0
