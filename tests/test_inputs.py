"""The seeded input generator: determinism, bf16 rounding, workload shapes."""
import numpy as np
import torch

import moe_inputs as mi


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    a = np.concatenate([g.standard_normal(100000).astype(np.float32) * 7,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 65504.0], np.float32)])
    want = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mi.f32_to_bf16_bits(a), want)
    np.testing.assert_array_equal(mi.bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_draws_are_deterministic_and_chunked():
    a = mi.draw_bf16((3, (1 << 22) + 5), 0, 1)
    b = mi.draw_bf16((3, (1 << 22) + 5), 0, 1)
    np.testing.assert_array_equal(a, b)
    c = mi.draw_bf16((3, (1 << 22) + 5), 1, 1)
    assert (a != c).mean() > 0.9


def test_tiny_shapes_and_scales():
    inp = mi.make_inputs("tiny")
    cfg = inp["cfg"]
    assert inp["x"].shape == (256, 512) and inp["x"].dtype == np.uint16
    assert inp["w_lat"].shape == (3072, 512)
    assert inp["w_head"].shape == (16, 3072)
    assert inp["w_gate"].shape == (16, 128, 512) and inp["w_down"].shape == (16, 512, 128)
    assert inp["bias"] is None
    w = mi.bf16_bits_to_f32(inp["w_gate"]).astype(np.float64)
    assert abs(w.std() * np.sqrt(cfg.d) - 1) < 0.01
    x = mi.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    assert abs(x.std() - 1) < 0.01


def test_workload_table():
    c = mi.CONFIGS
    assert c["frame"].T == 1792 and c["chunk"].T == 11392 and c["clip"].T == 107520 and c["refiner"].T == 48960
    assert all(v.n_heads == 12 and v.head_dim == 256 and v.top_k == 6 for v in c.values())


def test_zipf_shares_and_bias():
    q = mi.zipf_capped_shares(128, 1.2, 6)
    assert abs(q.sum() - 1) < 1e-12 and abs(q[0] - 1 / 6) < 1e-12 and np.all(np.diff(q) <= 0)
    assert 8.5e-4 < q[-1] < 9.5e-4
    b = mi.router_bias(mi.CONFIGS["clip"])
    assert b.shape == (128,) and b.dtype == np.float32 and b.max() == 0.0
    np.testing.assert_array_equal(b, mi.router_bias(mi.CONFIGS["clip"]))


def test_modality_scales():
    s = mi.x_row_scales(mi.CONFIGS["chunk"])
    assert s.shape == (11392,) and s[0] == 1.0 and s[10752] == 0.5 and s[-1] == np.float32(0.8)
