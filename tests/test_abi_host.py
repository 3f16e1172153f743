"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-side checks reject bad arguments before any CUDA call."""
import ctypes

import pytest

import fine_grained_moe_02_b300 as moe
from fine_grained_moe_02_b300 import binding as B


@pytest.fixture(scope="module")
def L():
    from fine_grained_moe_02_b300 import build
    build.build()
    return moe.lib()


def test_every_header_function_is_exported(L):
    names = moe.header_functions()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(B._SIGS), "binding signatures out of sync with include/moe.h"


def test_status_strings(L):
    assert moe.status_string(0) == "MOE_OK"
    assert moe.status_string(-4) == "MOE_ERR_WORKSPACE_TOO_SMALL"
    assert moe.status_string(12345) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("kw,ok", [
    (dict(T=256, d=512, E=16, inter=128), True),
    (dict(T=107520, d=4096, E=128, inter=1024), True),
    (dict(T=48960, d=4096, E=256, inter=512), True),
    (dict(T=1, d=64, E=8, inter=64, top_k=8), True),
    (dict(T=0, d=512, E=16, inter=128), False),
    (dict(T=256, d=500, E=16, inter=128), False),
    (dict(T=256, d=512, E=16, inter=100), False),
    (dict(T=256, d=512, E=257, inter=128), False),
    (dict(T=256, d=512, E=4, inter=128, top_k=6), False),
    (dict(T=256, d=512, E=16, inter=128, top_k=9), False),
    (dict(T=256, d=512, E=16, inter=128, n_heads=12, head_dim=100), False),
    (dict(T=400_000_000, d=512, E=16, inter=128), False),
])
def test_check_dims(L, kw, ok):
    d = moe.moe_dims.make(**kw)
    rc = moe.moe_check_dims(d)
    assert (rc == 0) == ok, (kw, rc)
    if not ok:
        assert rc == B.MOE_ERR_UNSUPPORTED_SHAPE


def test_workspace_sizes(L):
    d = moe.moe_dims.make(107520, 4096, 128, 1024)
    s, w, h = moe.moe_scratch_size(d), moe.moe_workspace_size(d), moe.moe_workspace_size_host(d)
    Tk = 107520 * 6
    assert s >= 107520 * 6144 * 2
    assert w >= s + Tk * 4096 * 2 + Tk * 1024 * 2 + 4 * Tk * 4
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_size(moe.moe_dims.make(0, 4096, 128, 1024))


@pytest.mark.parametrize("T,chunk", [(1, 1), (8192, 8192), (8193, 4097), (20000, 6667), (65536, 8192),
                                     (65537, 8193), (107520, 13440)])
def test_host_workspace_is_one_chunk_plus_staging(L, T, chunk):
    # moe_forward_host runs n = min(ceil(T / 8192), 8) chunks of ceil(T / n)
    # tokens: its workspace is one chunk's forward workspace plus x and out
    # staging for the whole batch (each rounded up to 1 KiB).
    d = 4096
    h = moe.moe_workspace_size_host(moe.moe_dims.make(T, d, 128, 1024))
    inner = moe.moe_workspace_size(moe.moe_dims.make(chunk, d, 128, 1024))
    io = -(-T * d * 2 // 1024) * 1024
    assert h == inner + 2 * io


def test_null_and_misaligned_pointers_are_rejected_on_the_host(L):
    d = moe.moe_dims.make(256, 512, 16, 128)
    P = ctypes.c_void_p
    ok, bad = P(0x10000), P(0x10001)
    nul = None
    # NULL required pointer
    assert L.moe_route(ctypes.byref(d), nul, ok, ok, nul, ok, ok, nul, ok, 1 << 30, nul) == B.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(ctypes.byref(d), ok, nul, ok, ok, ok, ok, ok, 1 << 30, nul) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(d), ok, ok, nul, ok, nul) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward(ctypes.byref(d), ok, ok, ok, nul, ok, ok, ok, nul, 1 << 30, nul) == B.MOE_ERR_INVALID_ARG
    # misaligned pointer
    assert L.moe_route(ctypes.byref(d), bad, ok, ok, nul, ok, ok, nul, ok, 1 << 30, nul) == B.MOE_ERR_MISALIGNED
    assert L.moe_expert_ffn(ctypes.byref(d), ok, ok, ok, ok, ok, bad, ok, 1 << 30, nul) == B.MOE_ERR_MISALIGNED
    assert L.moe_combine(ctypes.byref(d), ok, ok, ok, bad, nul) == B.MOE_ERR_MISALIGNED
    # workspace too small
    assert L.moe_dispatch(ctypes.byref(d), ok, ok, ok, ok, ok, ok, ok, 64, nul) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_forward(ctypes.byref(d), ok, ok, ok, nul, ok, ok, ok, ok, 64, nul) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # bad dims
    d0 = moe.moe_dims.make(256, 500, 16, 128)
    assert L.moe_route(ctypes.byref(d0), ok, ok, ok, nul, ok, ok, nul, ok, 1 << 30, nul) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_check_dims(None) == B.MOE_ERR_INVALID_ARG


def test_selftest_argument_checks(L):
    P = ctypes.c_void_p(0x10000)
    assert L.moe_selftest_timeout(None, 1 << 20, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_timeout(P, 1 << 20, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_timeout(ctypes.c_void_p(0x10008), 1 << 20, 1000, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_selftest_timeout(P, 4096, 1000, None) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_selftest_timeout_fused(None, 1 << 20, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_timeout_fused(P, 1 << 20, 10 ** 7 + 1, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_timeout_fused(ctypes.c_void_p(0x10008), 1 << 20, 1000, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_selftest_timeout_fused(P, 96 << 10, 1000, None) == B.MOE_ERR_WORKSPACE_TOO_SMALL


def test_undersized_tensors_are_rejected_before_any_device_work():
    # the C ABI takes bare pointers; the binding checks every buffer against dims
    import torch
    d = moe.moe_dims.make(256, 512, 16, 128, top_k=2)
    T, D, E, I, k, L = 256, 512, 16, 128, 2, 12 * 256
    bf = lambda n: torch.zeros(n, dtype=torch.bfloat16)
    ok = dict(x=bf(T * D), w_lat=bf(L * D), w_head=bf(E * L), w13=bf(E * 2 * I * D), w_down=bf(E * D * I),
              out=bf(T * D))
    for name in ok:
        args = dict(ok)
        args[name] = bf(ok[name].numel() - 1)
        with pytest.raises(ValueError, match=name):
            moe.moe_forward(d, args["x"], args["w_lat"], args["w_head"], None, args["w13"], args["w_down"],
                            args["out"], torch.zeros(1, dtype=torch.uint8))
    with pytest.raises(ValueError, match="act"):
        moe.moe_expert_gemm1(d, bf(T * k * D), torch.zeros(E + 1, dtype=torch.int32), bf(E * 2 * I * D),
                             bf(T * k * I - 8), torch.zeros(1, dtype=torch.uint8))
    with pytest.raises(ValueError, match="offsets"):
        moe.moe_dispatch(d, bf(T * D), torch.zeros(T * k, dtype=torch.int32), torch.zeros(E, dtype=torch.int32),
                         torch.zeros(T * k, dtype=torch.int32), torch.zeros(T * k, dtype=torch.int32),
                         bf(T * k * D), torch.zeros(1, dtype=torch.uint8))
    # shared experts: w13 holds E + n_shared experts, the slots top_k + n_shared
    ext = moe.moe_ext.make(n_shared=1)
    with pytest.raises(ValueError, match="w13"):
        moe.moe_forward_ext(d, ext, ok["x"], ok["w_lat"], ok["w_head"], None, ok["w13"], bf((E + 1) * D * I),
                            ok["out"], torch.zeros(1, dtype=torch.uint8))
    # head-local: per-head routers and experts
    h = moe.moe_dims.make(64, 256, 8, 64, top_k=2, n_heads=2, head_dim=128)
    with pytest.raises(ValueError, match="w_router"):
        moe.moe_forward_headlocal(h, bf(64 * 256), bf(2 * 8 * 128 - 1), None, bf(2 * 8 * 128 * 128),
                                  bf(2 * 8 * 128 * 64), bf(64 * 256), None, None, torch.zeros(1, dtype=torch.uint8))


@pytest.mark.parametrize("kw", [dict(router="two_stage"), dict(fuse=4), dict(router="folded", fuse=1)])
def test_layer_wrapper_rejects_unknown_options_before_any_device_work(kw):
    import torch
    dims = moe.moe_dims.make(256, 512, 16, 128, 6)
    w = torch.empty(1, dtype=torch.bfloat16)   # never touched: the options are checked first
    with pytest.raises(ValueError):
        moe.MoeLayer(dims, w, w, None, w, w, w, device="cpu", **kw)
