"""Sorting stage on the GPU vs the oracle's counting sort: bit-exact."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _run(T, d, E, k, idx_np, x_u16=None):
    dims = moe.moe_dims.make(T, d, E, 64, k, n_heads=1, head_dim=256)
    ws = moe.alloc_workspace(moe.moe_scratch_size(dims))
    if x_u16 is None:
        x_u16 = np.random.default_rng(T).integers(0, 1 << 16, size=(T, d), dtype=np.uint16) & np.uint16(0x7F7F)
    x = G.dev_bf16(x_u16)
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    row_of = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    src = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(dims, x, idx, offsets, row_of, src, x_perm, ws)
    status = moe.moe_get_device_status(ws)
    return status, offsets.cpu().numpy(), row_of.cpu().numpy(), src.cpu().numpy(), G.bits(x_perm), x_u16


def _random_idx(g, T, E, k):
    return np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,d,E,k", [
    (1, 64, 8, 6), (31, 128, 8, 1), (2047, 64, 16, 6), (2048, 64, 16, 6), (2049, 256, 128, 6),
    (5000, 64, 256, 8), (6000, 512, 6, 6), (300, 4096, 128, 6),
])
def test_dispatch_bit_exact(T, d, E, k):
    g = np.random.default_rng(T * 131 + E)
    idx = _random_idx(g, T, E, k)
    status, off, row_of, src, xp, x = _run(T, d, E, k, idx)
    assert status == 0
    G.check_dispatch(idx, E, off, row_of, src)
    np.testing.assert_array_equal(xp, x[src])


def test_dispatch_skewed_and_empty_groups():
    T, d, E, k = 4100, 64, 64, 6
    idx = np.tile(np.array([5, 17, 3, 60, 9, 33], np.int32), (T, 1))
    idx[::7] = np.array([0, 1, 2, 3, 4, 5])
    status, off, row_of, src, xp, x = _run(T, d, E, k, idx)
    assert status == 0
    G.check_dispatch(idx, E, off, row_of, src)
    np.testing.assert_array_equal(xp, x[src])
    assert off[-1] == T * k and (np.diff(off) == 0).sum() >= E - 12


def test_dispatch_flags_bad_ids_without_faulting():
    T, d, E, k = 100, 64, 16, 6
    g = np.random.default_rng(0)
    idx = _random_idx(g, T, E, k)
    idx[3, 2] = 16
    idx[50, 0] = -1
    idx[70, 4] = idx[70, 1]          # duplicate inside one token
    status, off, row_of, src, xp, x = _run(T, d, E, k, idx)
    assert status & moe.binding.MOE_DEV_BAD_EXPERT_ID
    assert row_of[3, 2] == -1 and row_of[50, 0] == -1 and row_of[70, 4] == -1
    assert off[-1] == T * k - 3
    # every other pair is placed exactly as the oracle places the valid pairs
    for t in range(T):
        for s in range(k):
            if row_of[t, s] >= 0:
                e = idx[t, s]
                assert off[e] <= row_of[t, s] < off[e + 1] and src[row_of[t, s]] == t
