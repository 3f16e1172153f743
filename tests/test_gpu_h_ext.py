"""Shared and modality-specific experts (moe_route_ext / moe_forward_ext) vs
the oracle's forward_ext."""
import numpy as np
import pytest
import torch

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _ext_inputs(**kw):
    cfg = mi.custom_config("ext", **kw)
    inp = mi.make_inputs(cfg)
    return inp


def test_ext_without_modalities_or_shared_equals_plain_forward():
    inp = mi.make_inputs("tiny")
    dev = G.Dev(inp)
    a = dev.forward()
    b = dev.forward_ext()
    assert dev.status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("kw", [
    dict(T=600, d=512, E=24, inter=128, top_k=2, modality_split=((300, 1.0), (200, 0.5), (100, 0.8)),
         modality_experts=((0, 8), (8, 16), (16, 24)), n_shared=1),
    dict(T=257, d=256, E=16, inter=64, top_k=6, modality_split=((200, 1.0), (57, 0.5)),
         modality_experts=((0, 10), (10, 16)), n_shared=2),
    dict(T=130, d=512, E=32, inter=128, top_k=4, n_shared=1),            # shared only
    dict(T=130, d=512, E=32, inter=128, top_k=4, modality_split=((100, 1.0), (30, 1.0)),
         modality_experts=((0, 16), (16, 32))),                          # modality ranges only
])
def test_ext_matches_oracle(kw):
    inp = _ext_inputs(**kw)
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, gate, logits = dev.route_ext()
    out = dev.forward_ext()
    assert dev.status() == 0
    idx_np = idx.cpu().numpy()
    G.check_routing_ext(inp, G.oracle_logits(inp), idx_np, gate.cpu().numpy(), logits.cpu().numpy())
    ref = O.forward_bits(inp, topk_idx=idx_np[:, :cfg.top_k])
    G.check_out(G.host_f64(out), ref["out"])


def test_ext_bad_modality_is_flagged():
    inp = _ext_inputs(T=64, d=256, E=16, inter=64, top_k=2, modality_split=((32, 1.0), (32, 1.0)),
                      modality_experts=((0, 8), (8, 16)), n_shared=1)
    inp["modality"][5] = 7
    dev = G.Dev(inp)
    idx, gate, _ = dev.route_ext()
    assert dev.status() & moe.binding.MOE_DEV_BAD_MODALITY
    assert np.all(idx.cpu().numpy()[5, :2] == -1)


def test_chunk_workload_with_modality_experts_and_a_shared_expert():
    inp = mi.make_inputs("chunk_mm")
    cfg = inp["cfg"]
    dev = G.Dev(inp)
    idx, gate, logits = dev.route_ext()
    out = dev.forward_ext()
    assert dev.status() == 0
    # sampled tokens from every modality: 96 video, all 256 text, all 384 audio rows are covered in part
    tok = np.sort(np.concatenate([mi.sample_tokens(10752, 96, seed=3), 10752 + mi.sample_tokens(256, 48, seed=4),
                                  11008 + mi.sample_tokens(384, 48, seed=5)]))
    idx_np = idx.cpu().numpy()[tok]
    G.check_routing_ext(inp, G.oracle_logits(inp, tok), idx_np, gate.cpu().numpy()[tok],
                        logits[torch.from_numpy(tok).cuda()].cpu().numpy(), tokens=tok)
    ref = O.forward_bits(inp, tokens=tok, topk_idx=idx_np[:, :cfg.top_k])
    G.check_out(G.host_f64(out[torch.from_numpy(tok).cuda()]), ref["out"])
