"""Gate-weighted combine on the GPU vs the oracle's fp64 combine."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,d,E,k", [(1, 64, 8, 6), (257, 512, 16, 6), (3000, 4096, 128, 6), (999, 128, 8, 8),
                                     (64, 64, 4, 1)])
def test_combine_matches_oracle(T, d, E, k):
    g = np.random.default_rng(T + d)
    idx = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, _, row_of, _ = O.dispatch(idx, E)
    y32 = g.standard_normal((T * k, d)).astype(np.float32)
    yb = torch.from_numpy(y32).to(torch.bfloat16)
    gate = g.random((T, k)).astype(np.float32)
    gate /= gate.sum(1, keepdims=True)
    dims = moe.moe_dims.make(T, d, E, 64, k, n_heads=1, head_dim=256)
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(dims, yb.cuda(), torch.from_numpy(row_of.astype(np.int32)).cuda(),
                    torch.from_numpy(gate).cuda(), out)
    ref = O.combine(yb.double().numpy(), row_of, gate.astype(np.float64))
    got = G.host_f64(out)
    # fp32 accumulation then one bf16 rounding: |err| <= 2^-8 |ref| + tiny
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)
