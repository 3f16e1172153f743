"""moe_dispatch_noalloc: the sorting stage for callers that cannot allocate
device memory (host frameworks that own all device memory and forbid
allocation while enqueueing work, latency-critical loops that cannot take an
allocation's device synchronisation).  Its scratch is a fixed array inside
libmoe, so its results must equal moe_dispatch's, call after call, although
the array keeps whatever the previous call left in it.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
from fine_grained_moe_02_b300 import binding as B
from tests import gpu_util as G


def _inputs(T, d, E, k, seed):
    g = np.random.default_rng(seed)
    idx = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = g.integers(0, 1 << 16, size=(T, d), dtype=np.uint16) & np.uint16(0x7F7F)
    return idx, x


def _outputs(T, d, E, k):
    return (torch.full((E + 1,), -9, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -9, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -9, dtype=torch.int32, device="cuda"),
            torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.gpu
def test_noalloc_dispatch_equals_workspace_dispatch_on_consecutive_calls():
    # different problems in a row: each must not see the previous one's
    # leftovers, a smaller one after a larger one and then a larger one again
    # (more counter cells than either before it), the last without a status word
    for (T, d, E, k, seed) in [(9000, 256, 128, 6, 1), (3001, 128, 64, 8, 2), (20000, 128, 256, 6, 4)]:
        idx_np, x_np = _inputs(T, d, E, k, seed)
        dims = moe.moe_dims.make(T, d, E, 64, k, n_heads=1, head_dim=256)
        x, idx = G.dev_bf16(x_np), torch.from_numpy(idx_np).cuda()
        ws = moe.alloc_workspace(moe.moe_scratch_size(dims))
        ref = _outputs(T, d, E, k)
        moe.moe_dispatch(dims, x, idx, *ref, ws)
        got = _outputs(T, d, E, k)
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if T != 20000 else None
        moe.moe_dispatch_noalloc(dims, x, idx, *got, status=status)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        assert status is None or int(status.item()) == 0
        for a, b in zip(ref, got):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
        G.check_dispatch(idx_np, E, got[0].cpu().numpy(), got[1].cpu().numpy(), got[2].cpu().numpy())


@pytest.mark.gpu
def test_noalloc_dispatch_reports_bad_ids_into_the_callers_status_word():
    T, d, E, k = 100, 64, 16, 6
    idx_np, x_np = _inputs(T, d, E, k, 3)
    idx_np[7, 1] = 99
    dims = moe.moe_dims.make(T, d, E, 64, k, n_heads=1, head_dim=256)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _outputs(T, d, E, k)
    moe.moe_dispatch_noalloc(dims, G.dev_bf16(x_np), torch.from_numpy(idx_np).cuda(), *out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & B.MOE_DEV_BAD_EXPERT_ID
    assert int(out[1][7, 1].item()) == -1


def test_noalloc_dispatch_rejects_problems_beyond_its_fixed_scratch():
    # ceil(T / 2048) * E must stay <= 65536; checked on the host before any CUDA call
    L = moe.lib()
    P = ctypes.c_void_p(0x10000)
    too_big = moe.moe_dims.make(2048 * 257, 64, 256, 64, 6)
    assert L.moe_dispatch_noalloc(ctypes.byref(too_big), P, P, P, P, P, P, None, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_dispatch_noalloc(ctypes.byref(too_big), None, P, P, P, P, P, None, None) == B.MOE_ERR_INVALID_ARG
