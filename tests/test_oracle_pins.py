"""The fp64 oracle against its pins, and planted mistakes against the pins.

CPU only.  A planted mistake is applied to a private copy of the oracle
module (never to the CUDA path); each must make at least one pin fail.
"""
import importlib.util
import pathlib

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import moe_oracle
from tests import oracle_pins as P

ORACLE_SRC = pathlib.Path(moe_oracle.__file__)


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin):
    pin(moe_oracle)


def _copy():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_SRC)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _m_bias_dropped(m):
    f = m.head_scores
    m.head_scores = lambda h, w, b, H, Dh: f(h, w, None, H, Dh)


def _m_first_head_only(m):
    def hs(h, w_head, bias, H, Dh):
        s = h[:, :Dh] @ w_head[:, :Dh].T
        return s if bias is None else s + bias
    m.head_scores = hs


def _m_wlat_not_transposed(m):
    m.latent_projection = lambda x, w: x @ w


def _m_ties_to_highest(m):
    def tk(p, k):
        E = p.shape[1]
        order = np.argsort(-p[:, ::-1], axis=1, kind="stable")
        return (E - 1 - order[:, :k]).astype(np.int32)
    m.topk_select = tk


def _m_gates_not_renormalised(m):
    m.renormalised_gates = lambda p, idx: np.take_along_axis(p, idx.astype(np.int64), 1)


def _m_silu_is_sigmoid(m):
    m.silu = lambda z: expit(z)


def _m_silu_on_up(m):
    def ffn(x_perm, offsets, wg, wu, wd, widen=None):
        return moe_oracle.expert_ffn(x_perm, offsets, wu, wg, wd, widen)
    m.expert_ffn = ffn


def _m_groups_reversed(m):
    """Rows inside each expert group in decreasing token order."""
    f = m.dispatch

    def disp(idx, E):
        counts, offsets, row_of, src = f(idx, E)
        src2 = src.copy()
        for e in range(E):
            lo, hi = offsets[e], offsets[e + 1]
            src2[lo:hi] = src[lo:hi][::-1]
        row2 = np.empty_like(row_of)
        for e in range(E):
            lo, hi = offsets[e], offsets[e + 1]
            for r in range(lo, hi):
                t = src2[r]
                s = int(np.nonzero(idx[t] == e)[0][0])
                row2[t, s] = r
        return counts, offsets, row2, src2
    m.dispatch = disp


def _m_combine_ignores_gates(m):
    f = m.combine
    m.combine = lambda y, row_of, gates: f(y, row_of, np.ones_like(gates))


def _m_softmax_wrong_axis(m):
    def sm(s):
        with np.errstate(invalid="ignore", over="ignore"):   # the mutant may meet inf - inf
            z = s - s.max(axis=0, keepdims=True)
            ez = np.exp(z)
            return ez / ez.sum(axis=0, keepdims=True)
    m.softmax = sm


def _m_widen_shift(m):
    m.widen_bf16 = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)


def _m_ext_mask_ignored(m):
    m.modality_mask = lambda modality, ranges, E: np.ones((len(modality), E), dtype=bool)


def _m_ext_shared_gated(m):
    f = m.swiglu_ffn
    m.swiglu_ffn = lambda x, wg, wu, wd: 0.5 * f(x, wg, wu, wd)


def _m_headlocal_wrong_slice(m):
    f = m.forward_headlocal

    def hl(x, w_router, bias, w_gate, w_up, w_down, n_heads, head_dim, k, **kw):
        return f(np.roll(x, head_dim, axis=1), w_router, bias, w_gate, w_up, w_down, n_heads, head_dim, k, **kw)
    m.forward_headlocal = hl


MUTANTS = [_m_headlocal_wrong_slice, _m_ext_mask_ignored, _m_ext_shared_gated, _m_bias_dropped, _m_first_head_only, _m_wlat_not_transposed, _m_ties_to_highest,
           _m_gates_not_renormalised, _m_silu_is_sigmoid, _m_silu_on_up, _m_groups_reversed,
           _m_combine_ignores_gates, _m_softmax_wrong_axis, _m_widen_shift]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutate):
    m = _copy()
    mutate(m)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(m)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught {mutate.__name__}"


def test_package_exports():
    for name in ["route", "dispatch", "gather", "expert_ffn", "combine", "forward", "forward_bits"]:
        assert callable(getattr(oracle, name))
