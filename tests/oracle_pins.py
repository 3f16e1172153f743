"""Pins for the fp64 oracle, written as plain functions of the oracle module.

Each ``pin_*`` raises AssertionError when the given oracle module disagrees
with something fixed independently of it: a hand-worked example in closed
form, brute force over all expert subsets, a library routine taking a
different route to the same quantity, or an invariant of the definition.
``test_oracle_pins.py`` runs them on the real oracle (all must hold) and on
planted-mistake copies of it (at least one must fail for each mistake).
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import scipy.special

RTOL = 1e-12


def _sig(z: float) -> float:
    return 1.0 / (1.0 + math.exp(-z))


# ----------------------------------------------------------------------------
# Hand-worked example (derived by hand from the layer definition).
# d=2, one head of dim 2, W_lat = I, E=2, W_head = I, no bias, inter=1.
#   expert 0: Wg=[1,0] Wu=[1,1] Wd=[1,2]^T ; expert 1: Wg=[0,1] Wu=[1,-1] Wd=[-1,1]^T
# Logits equal x.  silu(z) = z*sig(z).
#   x=[1,0],k=1: expert 0, gate 1; g=1,u=1 -> act=sig(1); out = sig(1)*[1,2]
#   x=[1,0],k=2: gates softmax([1,0]) = [sig(1), 1-sig(1)]; expert 1: g=0 -> act 0
#                out = sig(1) * sig(1)*[1,2]
#   x=[2,-1],k=2: gates [sig(3), 1-sig(3)]; e0: g=2,u=1 -> 2 sig(2);
#                e1: g=-1,u=3 -> -3 sig(-1); out = sig(3)*2sig(2)*[1,2]
#                + (1-sig(3))*(-3 sig(-1))*[-1,1]
#   x=[1,1],k=1: tie s=[1,1] -> expert 0; g=1,u=2 -> 2 sig(1); out = 2 sig(1)*[1,2]
# ----------------------------------------------------------------------------

HAND = dict(
    w_lat=np.eye(2), w_head=np.eye(2), bias=None,
    w_gate=np.array([[[1.0, 0.0]], [[0.0, 1.0]]]),      # [E=2, inter=1, d=2]
    w_up=np.array([[[1.0, 1.0]], [[1.0, -1.0]]]),
    w_down=np.array([[[1.0], [2.0]], [[-1.0], [1.0]]]),  # [E=2, d=2, inter=1]
)


def hand_cases():
    s1, s2, s3 = _sig(1.0), _sig(2.0), _sig(3.0)
    sm1 = _sig(-1.0)
    return [
        # x, k, idx, gates, out
        ([1.0, 0.0], 1, [0], [1.0], [s1, 2 * s1]),
        ([1.0, 0.0], 2, [0, 1], [s1, 1 - s1], [s1 * s1, 2 * s1 * s1]),
        ([2.0, -1.0], 2, [0, 1], [s3, 1 - s3],
         [s3 * 2 * s2 + (1 - s3) * (-3 * sm1) * -1.0, s3 * 2 * s2 * 2 + (1 - s3) * (-3 * sm1)]),
        ([1.0, 1.0], 1, [0], [1.0], [2 * s1, 4 * s1]),
    ]


def pin_hand_example(o):
    for x, k, idx, gates, out in hand_cases():
        r = o.forward(np.array([x]), HAND["w_lat"], HAND["w_head"], None,
                      HAND["w_gate"], HAND["w_up"], HAND["w_down"], 1, 2, k)
        assert list(r["topk_idx"][0]) == idx, (x, k, r["topk_idx"])
        np.testing.assert_allclose(r["gates"][0], gates, rtol=RTOL, atol=1e-15)
        np.testing.assert_allclose(r["out"][0], out, rtol=RTOL, atol=1e-15)


def pin_hand_permutation(o):
    """Tokens [1,0], [2,-1], [1,1] with k=1 all pick expert 0:
    offsets [0,3,3], src_token [0,1,2], row_of [[0],[1],[2]]."""
    x = np.array([[1.0, 0.0], [2.0, -1.0], [1.0, 1.0]])
    r = o.forward(x, HAND["w_lat"], HAND["w_head"], None, HAND["w_gate"], HAND["w_up"],
                  HAND["w_down"], 1, 2, 1)
    assert list(r["offsets"]) == [0, 3, 3]
    assert list(r["src_token"]) == [0, 1, 2]
    assert list(r["row_of"].ravel()) == [0, 1, 2]
    s1, s2 = _sig(1.0), _sig(2.0)
    want = [[s1, 2 * s1], [2 * s2, 4 * s2], [2 * s1, 4 * s1]]
    np.testing.assert_allclose(r["out"], want, rtol=RTOL)


# ----------------------------------------------------------------------------
# top-k: brute force over all subsets (max sum; lexicographically smallest
# sorted index tuple among equal sums == "ties to the lowest expert index")
# ----------------------------------------------------------------------------

def brute_topk_set(v: np.ndarray, k: int):
    best, best_sum = None, -math.inf
    for c in itertools.combinations(range(len(v)), k):   # lexicographic order
        sm = float(sum(v[i] for i in c))
        if sm > best_sum:
            best, best_sum = c, sm
    return best


def pin_topk_bruteforce(o):
    g = np.random.default_rng(7)
    for trial in range(60):
        E = int(g.integers(1, 13))
        k = int(g.integers(1, min(6, E) + 1))
        if trial % 2:
            s = g.integers(-2, 3, size=(4, E)).astype(np.float64)   # many exact ties
        else:
            s = g.standard_normal((4, E))
        idx = o.topk_select(o.softmax(s), k)
        for t in range(s.shape[0]):
            want = brute_topk_set(s[t], k)
            assert tuple(sorted(int(i) for i in idx[t])) == want, (s[t], k, idx[t], want)
            vals = s[t][idx[t]]
            for a in range(k - 1):   # slot order: value desc, then index asc
                assert vals[a] > vals[a + 1] or (vals[a] == vals[a + 1] and idx[t][a] < idx[t][a + 1])


def pin_gates_closed_forms(o):
    g = np.random.default_rng(3)
    s = g.standard_normal((5, 9)) * 3
    p = o.softmax(s)
    np.testing.assert_allclose(p, scipy.special.softmax(s, axis=1), rtol=1e-13)
    # k = E: the renormalised gates are the full softmax, in slot order
    idx = o.topk_select(p, 9)
    gates = o.renormalised_gates(p, idx)
    np.testing.assert_allclose(gates, np.take_along_axis(scipy.special.softmax(s, axis=1), idx.astype(np.int64), 1),
                               rtol=1e-13)
    # k < E: softmax restricted to the chosen logits
    idx = o.topk_select(p, 3)
    gates = o.renormalised_gates(p, idx)
    chosen = np.take_along_axis(s, idx.astype(np.int64), 1)
    np.testing.assert_allclose(gates, scipy.special.softmax(chosen, axis=1), rtol=1e-13)
    assert np.all(np.abs(gates.sum(1) - 1.0) <= 1e-12)


def _tiny_router(g, T, d, n_heads, head_dim, E):
    x = g.standard_normal((T, d))
    w_lat = g.standard_normal((n_heads * head_dim, d))
    w_head = g.standard_normal((E, n_heads * head_dim))
    b = g.standard_normal(E)
    return x, w_lat, w_head, b


def pin_router_scalar_loops(o):
    """s[t,e] = sum_l W_head[e,l] * (sum_i W_lat[l,i] x[t,i]) + b[e], by scalar loops."""
    g = np.random.default_rng(11)
    for (T, d, H, Dh, E) in [(3, 4, 2, 2, 3), (2, 6, 3, 2, 5)]:   # first case: d == H*Dh
        x, w_lat, w_head, b = _tiny_router(g, T, d, H, Dh, E)
        s = o.head_scores(o.latent_projection(x, w_lat), w_head, b, H, Dh)
        for t in range(T):
            for e in range(E):
                acc = 0.0
                for l in range(H * Dh):
                    hl = 0.0
                    for i in range(d):
                        hl += w_lat[l, i] * x[t, i]
                    acc += w_head[e, l] * hl
                assert abs(s[t, e] - (acc + b[e])) <= 1e-12 * (1 + abs(acc))


def pin_router_folded(o):
    """Linearity: s = x (W_head W_lat)^T + b, a different association."""
    g = np.random.default_rng(5)
    x, w_lat, w_head, b = _tiny_router(g, 17, 24, 3, 8, 7)      # d == L == 24
    s = o.head_scores(o.latent_projection(x, w_lat), w_head, b, 3, 8)
    s2 = np.linalg.multi_dot([x, w_lat.T, w_head.T]) + b
    np.testing.assert_allclose(s, s2, rtol=1e-11, atol=1e-11)
    s3 = x @ (w_head @ w_lat).T + b
    np.testing.assert_allclose(s, s3, rtol=1e-11, atol=1e-11)


def pin_bias_forces_selection(o):
    """A large bias on experts {2, 4} makes every token pick them first (k=2)."""
    g = np.random.default_rng(9)
    x, w_lat, w_head, _ = _tiny_router(g, 6, 8, 2, 4, 6)
    b = np.zeros(6)
    b[4], b[2] = 200.0, 100.0
    s, idx, gates = o.route(x, w_lat, w_head, b, 2, 4, 2)
    assert np.all(idx[:, 0] == 4) and np.all(idx[:, 1] == 2)
    # gates depend on the biased logits: softmax of the two chosen biased logits
    chosen = np.take_along_axis(s, idx.astype(np.int64), 1)
    np.testing.assert_allclose(gates, scipy.special.softmax(chosen, 1), rtol=1e-12)
    s0 = o.head_scores(o.latent_projection(x, w_lat), w_head, None, 2, 4)
    np.testing.assert_allclose(s - s0, np.broadcast_to(b, s.shape), atol=1e-12)


# ----------------------------------------------------------------------------
# sorting
# ----------------------------------------------------------------------------

def _random_idx(g, T, E, k):
    return np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def pin_dispatch_invariants(o):
    g = np.random.default_rng(2)
    for (T, E, k) in [(1, 6, 6), (37, 8, 3), (200, 16, 6), (64, 6, 6), (5, 256, 6)]:
        idx = _random_idx(g, T, E, k)
        counts, offsets, row_of, src = o.dispatch(idx, E)
        assert counts.sum() == T * k
        assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) >= 0)
        np.testing.assert_array_equal(np.diff(offsets), counts)
        np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        assert sorted(row_of.ravel().tolist()) == list(range(T * k))   # bijection
        for t in range(T):
            for s in range(k):
                assert src[row_of[t, s]] == t
                e = idx[t, s]
                assert offsets[e] <= row_of[t, s] < offsets[e + 1]
        for e in range(E):                      # increasing token order in a group
            assert np.all(np.diff(src[offsets[e]:offsets[e + 1]]) > 0)


def pin_dispatch_vs_stable_sort(o):
    """The permutation equals a stable sort of (expert, token) pairs."""
    g = np.random.default_rng(4)
    T, E, k = 300, 32, 6
    idx = _random_idx(g, T, E, k)
    _, _, row_of, src = o.dispatch(idx, E)
    flat_e = idx.ravel().astype(np.int64)
    flat_t = np.repeat(np.arange(T), k)
    order = np.lexsort((flat_t, flat_e))          # primary key expert, then token
    np.testing.assert_array_equal(src, flat_t[order])
    rows = np.empty(T * k, dtype=np.int64)
    rows[order] = np.arange(T * k)
    np.testing.assert_array_equal(row_of.ravel(), rows)


def pin_dispatch_rejects_bad_ids(o):
    for bad in (-1, 8):
        try:
            o.dispatch(np.array([[0, bad]], dtype=np.int32), 8)
        except ValueError:
            continue
        raise AssertionError("out-of-range expert id accepted")


# ----------------------------------------------------------------------------
# calculation
# ----------------------------------------------------------------------------

def pin_silu_values(o):
    z = np.array([0.0, 1.0, -1.0, 2.0, -30.0, 30.0])
    want = [0.0, _sig(1.0), -_sig(-1.0), 2 * _sig(2.0), -30 * _sig(-30.0), 30 * _sig(30.0)]
    np.testing.assert_allclose(o.silu(z), want, rtol=1e-14, atol=1e-300)


def pin_single_expert_is_swiglu(o):
    """E = k = 1: the layer is a textbook SwiGLU FFN, written out with scalar loops."""
    g = np.random.default_rng(12)
    T, d, I = 3, 5, 4
    x = g.standard_normal((T, d))
    w_lat, w_head = g.standard_normal((2 * 2, d)), g.standard_normal((1, 4))
    wg, wu, wd = g.standard_normal((1, I, d)), g.standard_normal((1, I, d)), g.standard_normal((1, d, I))
    r = o.forward(x, w_lat, w_head, None, wg, wu, wd, 2, 2, 1)
    for t in range(T):
        act = []
        for j in range(I):
            gj = sum(wg[0, j, i] * x[t, i] for i in range(d))
            uj = sum(wu[0, j, i] * x[t, i] for i in range(d))
            act.append(gj * _sig(gj) * uj)
        for i in range(d):
            want = sum(wd[0, i, j] * act[j] for j in range(I))
            assert abs(r["out"][t, i] - want) <= 1e-12 * (1 + abs(want))
    assert np.all(r["gates"] == 1.0)


def pin_forward_direct(o):
    """The sorted path equals the per-token definition with no permutation:
    out[t] = sum_s gate[t,s] * FFN_{idx[t,s]}(x[t])."""
    g = np.random.default_rng(21)
    T, d, H, Dh, E, I, k = 23, 8, 2, 3, 7, 4, 3
    x = g.standard_normal((T, d))
    w_lat, w_head = g.standard_normal((H * Dh, d)), g.standard_normal((E, H * Dh))
    b = g.standard_normal(E)
    wg, wu, wd = g.standard_normal((E, I, d)), g.standard_normal((E, I, d)), g.standard_normal((E, d, I))
    r = o.forward(x, w_lat, w_head, b, wg, wu, wd, H, Dh, k)
    for t in range(T):
        acc = np.zeros(d)
        for s in range(k):
            e = r["topk_idx"][t, s]
            gg, uu = wg[e] @ x[t], wu[e] @ x[t]
            acc += r["gates"][t, s] * (wd[e] @ (gg * _sig_vec(gg) * uu))
        np.testing.assert_allclose(r["out"][t], acc, rtol=1e-12, atol=1e-12)


def _sig_vec(z):
    return np.array([_sig(float(v)) for v in z])


def pin_subset_rows(o):
    """The layer is per-token: a token subset gives the same output rows."""
    g = np.random.default_rng(31)
    T, d, H, Dh, E, I, k = 40, 8, 2, 4, 9, 4, 6
    x = g.standard_normal((T, d))
    w = (g.standard_normal((H * Dh, d)), g.standard_normal((E, H * Dh)), g.standard_normal(E),
         g.standard_normal((E, I, d)), g.standard_normal((E, I, d)), g.standard_normal((E, d, I)))
    full = o.forward(x, *w, H, Dh, k)
    sub = np.array([3, 4, 17, 39])
    part = o.forward(x[sub], *w, H, Dh, k)
    np.testing.assert_allclose(part["out"], full["out"][sub], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(part["topk_idx"], full["topk_idx"][sub])


def pin_combine_slot_sum(o):
    g = np.random.default_rng(8)
    y = g.standard_normal((12, 5))
    row_of = np.array([[3, 7], [0, 11], [5, 1]])
    gates = np.array([[0.25, 0.75], [1.0, 0.0], [0.5, 0.5]])
    out = o.combine(y, row_of, gates)
    for t in range(3):
        np.testing.assert_allclose(out[t], gates[t, 0] * y[row_of[t, 0]] + gates[t, 1] * y[row_of[t, 1]],
                                   rtol=1e-15)


def pin_widen_bf16(o):
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x4049, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -1.0, 0.0, -0.0, 3.140625, 3.3895313892515355e38, 9.183549615799121e-41]
    np.testing.assert_array_equal(o.widen_bf16(bits), np.array(want))


ALL_PINS = [
    pin_hand_example, pin_hand_permutation, pin_topk_bruteforce, pin_gates_closed_forms,
    pin_router_scalar_loops, pin_router_folded, pin_bias_forces_selection,
    pin_dispatch_invariants, pin_dispatch_vs_stable_sort, pin_dispatch_rejects_bad_ids,
    pin_silu_values, pin_single_expert_is_swiglu, pin_forward_direct, pin_subset_rows,
    pin_combine_slot_sum, pin_widen_bf16,
]


# ----------------------------------------------------------------------------
# shared and modality-specific experts
# ----------------------------------------------------------------------------

def _ext_case(g, T=30, d=8, H=2, Dh=4, E=9, I=4, S=1):
    x = g.standard_normal((T, d))
    w_lat, w_head = g.standard_normal((H * Dh, d)), g.standard_normal((E, H * Dh))
    b = g.standard_normal(E)
    wg, wu = g.standard_normal((E + S, I, d)), g.standard_normal((E + S, I, d))
    wd = g.standard_normal((E + S, d, I))
    return x, w_lat, w_head, b, wg, wu, wd


def pin_ext_reduces_to_plain_layer(o):
    """One modality covering every expert and no shared expert: the plain layer."""
    g = np.random.default_rng(41)
    x, w_lat, w_head, b, wg, wu, wd = _ext_case(g, S=0)
    a = o.forward(x, w_lat, w_head, b, wg, wu, wd, 2, 4, 3)
    e = o.forward_ext(x, w_lat, w_head, b, wg, wu, wd, 2, 4, 3, modality=np.zeros(len(x), int),
                      expert_ranges=((0, 9),), n_shared=0)
    np.testing.assert_array_equal(a["topk_idx"], e["topk_idx"])
    np.testing.assert_allclose(a["out"], e["out"], rtol=1e-13, atol=1e-13)


def pin_ext_modality_and_shared_by_definition(o):
    """Per token, by scalar loops: only the modality's experts compete, their
    softmax over the chosen k gives the gates, and the shared expert is added."""
    g = np.random.default_rng(43)
    T, k = 30, 2
    x, w_lat, w_head, b, wg, wu, wd = _ext_case(g, T=T)
    b[7] = 1e3                       # a huge bias on expert 7 must not leak into modality 0
    mod = np.array([t % 3 for t in range(T)])
    ranges = ((0, 4), (4, 7), (7, 9))
    r = o.forward_ext(x, w_lat, w_head, b, wg, wu, wd, 2, 4, k, modality=mod, expert_ranges=ranges, n_shared=1)
    for t in range(T):
        lo, hi = ranges[mod[t]]
        s = [sum(w_head[e, l] * sum(w_lat[l, i] * x[t, i] for i in range(8)) for l in range(8)) + b[e]
             for e in range(lo, hi)]
        order = sorted(range(hi - lo), key=lambda j: (-s[j], j))[:k]
        assert [lo + j for j in order] == list(r["topk_idx"][t])
        m = max(s[j] for j in order)
        w = [math.exp(s[j] - m) for j in order]
        acc = np.zeros(8)
        for wi, j in zip(w, order):
            e = lo + j
            acc += wi / sum(w) * (wd[e] @ (_sig_vec(wg[e] @ x[t]) * (wg[e] @ x[t]) * (wu[e] @ x[t])))
        acc += wd[9] @ (_sig_vec(wg[9] @ x[t]) * (wg[9] @ x[t]) * (wu[9] @ x[t]))
        np.testing.assert_allclose(r["out"][t], acc, rtol=1e-10, atol=1e-10)


def pin_ext_rejects_routing_outside_the_modality(o):
    g = np.random.default_rng(47)
    x, w_lat, w_head, b, wg, wu, wd = _ext_case(g, T=4)
    try:
        o.forward_ext(x, w_lat, w_head, b, wg, wu, wd, 2, 4, 1, modality=np.zeros(4, int),
                      expert_ranges=((0, 3), (3, 9)), n_shared=1, topk_idx=np.array([[5], [0], [1], [2]]))
    except ValueError:
        return
    raise AssertionError("routing outside the modality accepted")


ALL_PINS += [pin_ext_reduces_to_plain_layer, pin_ext_modality_and_shared_by_definition,
             pin_ext_rejects_routing_outside_the_modality]


# ----------------------------------------------------------------------------
# head-local MultiHead MoE
# ----------------------------------------------------------------------------

def _hl_case(g, T=20, H=3, Dh=4, E=5, I=3):
    x = g.standard_normal((T, H * Dh))
    wr = g.standard_normal((H, E, Dh))
    b = g.standard_normal((H, E))
    wg, wu = g.standard_normal((H, E, I, Dh)), g.standard_normal((H, E, I, Dh))
    wd = g.standard_normal((H, E, Dh, I))
    return x, wr, b, wg, wu, wd


def pin_headlocal_by_definition(o):
    """Per token and head, by scalar loops: the head's own slice scores its
    own experts; the k best (ties to the lowest index) are gated by their
    softmax; the head's slot of the output is their gate-weighted sum."""
    g = np.random.default_rng(51)
    T, H, Dh, E, k = 20, 3, 4, 5, 2
    x, wr, b, wg, wu, wd = _hl_case(g)
    r = o.forward_headlocal(x, wr, b, wg, wu, wd, H, Dh, k)
    for t in range(T):
        for j in range(H):
            xj = x[t, j * Dh:(j + 1) * Dh]
            s = [sum(wr[j, e, i] * xj[i] for i in range(Dh)) + b[j, e] for e in range(E)]
            order = sorted(range(E), key=lambda e: (-s[e], e))[:k]
            assert list(r["topk_idx"][j, t]) == order
            w = [math.exp(s[e] - s[order[0]]) for e in order]
            acc = np.zeros(Dh)
            for wi, e in zip(w, order):
                gg, uu = wg[j, e] @ xj, wu[j, e] @ xj
                acc += wi / sum(w) * (wd[j, e] @ (gg * _sig_vec(gg) * uu))
            np.testing.assert_allclose(r["out"][t, j * Dh:(j + 1) * Dh], acc, rtol=1e-11, atol=1e-11)


def pin_headlocal_heads_are_independent(o):
    """Changing one head's slice changes only that head's output columns."""
    g = np.random.default_rng(53)
    x, wr, b, wg, wu, wd = _hl_case(g)
    r1 = o.forward_headlocal(x, wr, b, wg, wu, wd, 3, 4, 2)
    x2 = x.copy()
    x2[:, 4:8] += g.standard_normal((x.shape[0], 4))
    r2 = o.forward_headlocal(x2, wr, b, wg, wu, wd, 3, 4, 2)
    np.testing.assert_array_equal(r1["out"][:, :4], r2["out"][:, :4])
    np.testing.assert_array_equal(r1["out"][:, 8:], r2["out"][:, 8:])
    assert np.abs(r1["out"][:, 4:8] - r2["out"][:, 4:8]).max() > 1e-6


ALL_PINS += [pin_headlocal_by_definition, pin_headlocal_heads_are_independent]
