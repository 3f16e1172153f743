"""Head-local MultiHead MoE (moe_forward_headlocal) vs the oracle's
forward_headlocal: each head's routing and the concatenated output."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


class HLDev:
    def __init__(self, inp):
        cfg = self.cfg = inp["cfg"]
        self.inp = inp
        self.dims = moe.moe_dims.make(cfg.T, cfg.d, cfg.E, cfg.inter, cfg.top_k, cfg.n_heads, cfg.head_dim)
        self.x = G.dev_bf16(inp["x"])
        self.w_router = G.dev_bf16(inp["w_router"])
        self.w_down = G.dev_bf16(inp["w_down"])
        self.w13 = torch.empty((cfg.n_heads, cfg.E, 2 * cfg.inter, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
        moe.moe_prepare_weights_headlocal(self.dims, G.dev_bf16(inp["w_gate"]), G.dev_bf16(inp["w_up"]), self.w13)
        self.ws = moe.alloc_workspace(moe.moe_workspace_size_headlocal(self.dims))

    def forward(self, staged=False):
        c = self.cfg
        out = torch.empty((c.T, c.d), dtype=torch.bfloat16, device="cuda")
        idx = torch.empty((c.n_heads, c.T, c.top_k), dtype=torch.int32, device="cuda")
        logits = torch.empty((c.n_heads, c.T, c.E), dtype=torch.float32, device="cuda")
        bias = None if self.inp["bias"] is None else torch.from_numpy(np.ascontiguousarray(self.inp["bias"])).cuda()
        moe.moe_forward_headlocal(self.dims, self.x, self.w_router, bias, self.w13, self.w_down, out, idx, logits,
                                  self.ws, staged=staged)
        return out, idx, logits


def _check(inp, out, idx, logits, tokens=None):
    cfg = inp["cfg"]
    idx_np = idx.cpu().numpy()
    lg = logits.cpu().numpy()
    if tokens is not None:
        idx_np, lg = idx_np[:, tokens], lg[:, tokens]
    ref = O.forward_bits(inp, tokens=tokens, topk_idx=idx_np)
    for j in range(cfg.n_heads):
        # each head's scores from the oracle; the layer returns no gates, so
        # the gate check is the oracle's own renormalisation of the GPU's ids
        s_ref = ref["logits"][j]
        gates = O.renormalised_gates(O.softmax(s_ref), idx_np[j])
        G.check_routing(s_ref, idx_np[j], gates.astype(np.float32), cfg.top_k, lg[j])
    got = G.host_f64(out if tokens is None else out[torch.from_numpy(tokens).cuda()])
    return G.check_out(got, ref["out"])


@pytest.mark.parametrize("kw", [
    dict(T=300, d=128, n_heads=2, head_dim=64, E=8, inter=64, top_k=2),
    dict(T=1000, d=512, n_heads=4, head_dim=128, E=32, inter=128, top_k=6),
    dict(T=129, d=768, n_heads=3, head_dim=256, E=256, inter=64, top_k=8),
    # 16 x 256 head-local experts exceed one grouped-GEMM launch: head by head
    dict(T=200, d=1024, n_heads=16, head_dim=64, E=256, inter=64, top_k=2),
])
def test_headlocal_matches_oracle(kw):
    inp = mi.make_inputs(mi.custom_config("hl", head_local=True, **kw))
    dev = HLDev(inp)
    out, idx, logits = dev.forward()
    assert moe.moe_get_device_status(dev.ws) == 0
    _check(inp, out, idx, logits)


def test_headlocal_workload_sampled():
    inp = mi.make_inputs("headlocal")
    dev = HLDev(inp)
    out, idx, logits = dev.forward()
    assert moe.moe_get_device_status(dev.ws) == 0
    tok = mi.sample_tokens(inp["cfg"].T, 192, seed=17)
    _check(inp, out, idx, logits, tokens=tok)
    # deterministic
    out2, _, _ = dev.forward()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_headlocal_per_head_router_bias():
    # a [n_heads, E] router bias moves each head's own selection and gates
    inp = mi.make_inputs(mi.custom_config("hlb", head_local=True, T=500, d=512, n_heads=4, head_dim=128, E=32,
                                          inter=64, top_k=4))
    rng = np.random.default_rng(8)
    inp["bias"] = rng.normal(0.0, 3.0, (4, 32)).astype(np.float32)
    dev = HLDev(inp)
    out, idx, logits = dev.forward()
    assert moe.moe_get_device_status(dev.ws) == 0
    _check(inp, out, idx, logits)
    # the bias is the only difference from the unbiased layer, and it changes the routing
    inp0 = dict(inp)
    inp0["bias"] = None
    _, idx0, _ = HLDev(inp0).forward()
    assert not torch.equal(idx, idx0)


@pytest.mark.parametrize("kw", [
    dict(T=300, d=128, n_heads=2, head_dim=64, E=8, inter=64, top_k=2),
    dict(T=1000, d=512, n_heads=4, head_dim=128, E=32, inter=128, top_k=6),
    dict(T=129, d=768, n_heads=3, head_dim=256, E=256, inter=64, top_k=8),
    dict(T=700, d=768, n_heads=3, head_dim=256, E=40, inter=512, top_k=6),
    dict(T=200, d=1024, n_heads=16, head_dim=64, E=256, inter=64, top_k=2),   # 4096 experts: staged head by head
    dict(T=900, d=256, n_heads=4, head_dim=64, E=16, inter=256, top_k=3),      # fused, 64-wide heads
    dict(T=640, d=384, n_heads=2, head_dim=192, E=24, inter=384, top_k=4),     # fused, 3 k-slices, 3 pieces
    dict(T=40, d=512, n_heads=2, head_dim=256, E=256, inter=128, top_k=2),     # fused, most groups empty
    dict(T=2500, d=512, n_heads=2, head_dim=256, E=4, inter=256, top_k=1),     # fused, groups of many tiles
    dict(T=300, d=1024, n_heads=16, head_dim=64, E=256, inter=128, top_k=2),   # fused over 4096 groups
])
def test_fused_expert_kernel_gives_the_staged_bits(kw):
    # the fused expert kernel rounds act to bf16 exactly where the separate
    # GEMMs do and runs the same MMA sequence: identical outputs
    inp = mi.make_inputs(mi.custom_config("hlf", head_local=True, **kw))
    dev = HLDev(inp)
    out, idx, _ = dev.forward()
    assert moe.moe_get_device_status(dev.ws) == 0
    ref, idx2, _ = dev.forward(staged=True)
    assert moe.moe_get_device_status(dev.ws) == 0
    assert torch.equal(idx, idx2)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    _check(inp, out, idx, _)


def test_fused_expert_kernel_wait_timeout_is_reported_and_the_context_survives():
    # the fused kernel's weight loader issues nothing: the tensor-core
    # thread's stage wait runs out after 20 ms, the other roles abort
    ws = moe.alloc_workspace(1 << 20)
    moe.moe_clear_device_status(ws)
    moe.moe_selftest_timeout_fused(ws, 20_000)
    assert moe.moe_get_device_status(ws) & moe.binding.MOE_DEV_TIMEOUT
    # the GPU still runs the fused kernel correctly afterwards (tensor memory was released)
    inp = mi.make_inputs(mi.custom_config("hlt", head_local=True, T=300, d=512, n_heads=2, head_dim=256, E=8,
                                          inter=256, top_k=2))
    dev = HLDev(inp)
    out, idx, logits = dev.forward()
    assert moe.moe_get_device_status(dev.ws) == 0
    _check(inp, out, idx, logits)
