"""Fixtures under tests/golden/:

* pages_routing.json: figures the source pages print for the routed layer
  (12 latent heads of 256 dims, top-6; the head-local variant's 256 experts
  per head), each with its page and passage.  Every page workload of the
  seeded input generator, and the library's shape rules, must take them.
* tiny_oracle.json: sampled fp64 oracle outputs of the tiny workload,
  written by tests/golden/make_golden.py (oracle/ only).  The oracle must
  still reproduce them; a GPU test compares moe_forward with them.
"""
import ctypes
import json
import pathlib

import numpy as np
import pytest

import fine_grained_moe_02_b300 as moe
import moe_inputs as mi
from fine_grained_moe_02_b300 import binding as B
from oracle import moe_oracle as O

GOLDEN = pathlib.Path(__file__).resolve().parent / "golden"
PAGE_WORKLOADS = ["frame", "chunk", "clip", "refiner", "chunk_mm"]   # latent-routed layer, the pages' geometry


def _facts():
    return {f["name"]: f["value"] for f in json.loads((GOLDEN / "pages_routing.json").read_text())["facts"]}


def test_every_fact_cites_a_page():
    for f in json.loads((GOLDEN / "pages_routing.json").read_text())["facts"]:
        assert f["source"].strip() and isinstance(f["value"], int), f


@pytest.mark.parametrize("name", PAGE_WORKLOADS)
def test_page_workloads_take_the_pages_routing(name):
    f, cfg = _facts(), mi.CONFIGS[name]
    assert (cfg.n_heads, cfg.head_dim, cfg.top_k) == (f["n_heads"], f["head_dim"], f["top_k"])
    assert cfg.n_heads * cfg.head_dim == f["latent_dim"]


def test_headlocal_workload_takes_the_pages_split():
    f, cfg = _facts(), mi.CONFIGS["headlocal"]
    assert cfg.head_local and (cfg.n_heads, cfg.head_dim, cfg.top_k) == (f["n_heads"], f["head_dim"], f["top_k"])
    assert cfg.d == f["latent_dim"] and cfg.E == f["headlocal_experts_per_head"]
    assert cfg.n_heads * cfg.top_k == f["headlocal_experts_per_token"]
    assert cfg.n_heads * cfg.E == f["headlocal_expert_units_per_layer"]


def test_library_shape_rules_take_the_pages_shapes():
    from fine_grained_moe_02_b300 import build
    build.build()
    L = moe.lib()
    f = _facts()
    clip = mi.CONFIGS["clip"]
    d = moe.moe_dims.make(clip.T, clip.d, clip.E, clip.inter, f["top_k"], f["n_heads"], f["head_dim"])
    assert L.moe_check_dims(ctypes.byref(d)) == B.MOE_OK
    hl = mi.CONFIGS["headlocal"]
    dh = moe.moe_dims.make(hl.T, f["latent_dim"], f["headlocal_experts_per_head"], hl.inter, f["top_k"],
                           f["n_heads"], f["head_dim"])
    n = ctypes.c_size_t(0)
    assert L.moe_workspace_size_headlocal(ctypes.byref(dh), ctypes.byref(n)) == B.MOE_OK and n.value > 0


def test_oracle_reproduces_the_stored_tiny_sample():
    g = json.loads((GOLDEN / "tiny_oracle.json").read_text())
    inp = mi.make_inputs("tiny")
    r = O.forward_bits(inp)
    t = g["tokens"]
    assert [int(v) for v in r["offsets"]] == g["offsets"]
    np.testing.assert_array_equal(r["topk_idx"][t], np.array(g["topk_idx"]))
    np.testing.assert_allclose(r["gates"][t], np.array(g["gates"]), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r["out"][t, :g["out_cols"]], np.array(g["out"]), rtol=1e-9, atol=1e-12)
