"""Pins for the oracle's route packing, grouped experts and additive stages
(exllamav3 #284 "Summary", "API contract"; TensorFold #837 "What this changes")."""

import numpy as np
import pytest
import scipy.special

from oracle import exl3_oracle as O
from workloads import make_projection, CB_MCG, CB_3INST, CB_MUL1


# ---------------------------------------------------------------- route pack
@pytest.mark.parametrize("M,topk,E,cap", [(16, 2, 8, 3), (37, 8, 19, 5), (1, 8, 192, 512),
                                          (64, 4, 5, 64), (0, 2, 4, 1)])
def test_route_pack_is_a_stable_counting_sort(M, topk, E, cap):
    ids = np.random.default_rng(M + E).integers(0, E, size=(M, topk))
    off, packed, tiles, nact = O.route_pack(ids, E, cap)
    flat = ids.reshape(-1)
    assert np.array_equal(packed, np.argsort(flat, kind="stable"))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert sorted(packed.tolist()) == list(range(M * topk))
    assert nact == len(np.unique(flat))
    # tiles: ascending expert, contiguous cover of each span, capacity-sized
    pos = 0
    for e in range(E):
        n = off[e + 1] - off[e]
        mine = tiles[tiles[:, 0] == e]
        assert len(mine) == -(-n // cap)
        for i, (_, start, ln) in enumerate(mine):
            assert start == off[e] + i * cap and 1 <= ln <= cap
            pos += ln
    assert pos == M * topk
    assert np.all(np.diff(tiles[:, 0]) >= 0)


def test_route_pack_counts_duplicates_and_rejects_bad_ids():
    ids = np.array([[3, 3], [1, 3]])
    off, packed, tiles, nact = O.route_pack(ids, 4, 2)
    assert off.tolist() == [0, 0, 1, 1, 4]
    assert packed.tolist() == [2, 0, 1, 3]
    assert tiles.tolist() == [[1, 0, 1], [3, 1, 2], [3, 3, 1]]
    with pytest.raises(ValueError):
        O.route_pack(np.array([[0, 4]]), 4, 2)
    with pytest.raises(ValueError):
        O.route_pack(np.array([[-1, 0]]), 4, 2)


# ---------------------------------------------------------------- experts
H, I, E = 256, 128, 4


def _experts(seed=0, cbs=(CB_MCG, CB_3INST, CB_MUL1, CB_MCG), Ks=(3, 4, 5, 2)):
    P = {}
    for e in range(E):
        for p in range(3):
            shp = (H, I) if p < 2 else (I, H)
            P[e, p] = make_projection([seed, e, p], *shp, Ks[e], cbs[e])
    return lambda e, p: P[e, p]


def test_silu_is_logistic_times_input():
    g = np.linspace(-30, 30, 121)
    assert np.allclose(O.silu(g), g * scipy.special.expit(g), rtol=1e-14, atol=1e-300)


def test_single_route_unit_weight_is_the_expert_chain():
    get = _experts()
    x = np.random.default_rng(1).standard_normal((3, H))
    ids = np.array([[2], [0], [2]])
    out = O.moe_forward(x, ids, np.ones((3, 1)), get)
    for t in range(3):
        e = ids[t, 0]
        g = O.linear(x[t:t + 1], get(e, 0))
        u = O.linear(x[t:t + 1], get(e, 1))
        d = O.linear(g / (1 + np.exp(-g)) * u, get(e, 2))
        assert np.allclose(out[t], d[0], rtol=1e-12, atol=1e-14)


def _with_scale_times(proj, factor):
    # a copy whose per-channel output scale is multiplied by an exact power of
    # two (so the fp16 scale stays exact): the projection's output times factor
    from dataclasses import replace
    return replace(proj, scale=(proj.scale.astype(np.float64) * factor).astype(np.float16))


def test_swiglu_gates_through_the_gate_projection():
    # SwiGLU = silu(gate) * up: the expert's output is linear in the up
    # projection, and SiLU's odd part is the identity (silu(g) - silu(-g) = g
    # because sigma(g) + sigma(-g) = 1), so negating the gate projection moves
    # the output by exactly down(gate(x) * up(x)).  A nonlinearity on the up
    # branch fails the first check; a missing one fails the second.
    get = _experts()
    x = np.random.default_rng(11).standard_normal((3, H))
    ids = np.array([[1], [3], [0]])
    rw = np.ones((3, 1))
    base = O.moe_forward(x, ids, rw, get)
    up2 = O.moe_forward(x, ids, rw, lambda e, p: _with_scale_times(get(e, p), -2.0) if p == 1 else get(e, p))
    assert np.allclose(up2, -2.0 * base, rtol=1e-11, atol=1e-12 * np.abs(base).max())
    neg = O.moe_forward(x, ids, rw, lambda e, p: _with_scale_times(get(e, p), -1.0) if p == 0 else get(e, p))
    for t in range(3):
        e = ids[t, 0]
        g = O.linear(x[t:t + 1], get(e, 0))
        u = O.linear(x[t:t + 1], get(e, 1))
        want = O.linear(g * u, get(e, 2))[0]
        assert np.allclose(base[t] - neg[t], want, rtol=1e-9, atol=1e-11 * np.abs(want).max())
        # and the gate side is not linear: negating it is not negating the output
        assert np.abs(neg[t] + base[t]).max() > 1e-3 * np.abs(base[t]).max()


def test_combine_is_linear_in_route_weights_and_counts_duplicates():
    get = _experts()
    x = np.random.default_rng(2).standard_normal((4, H))
    ids = np.array([[0, 1], [3, 3], [2, 0], [1, 2]])
    rw = np.random.default_rng(3).uniform(0.1, 0.9, size=(4, 2))
    out = O.moe_forward(x, ids, rw, get)
    assert np.allclose(O.moe_forward(x, ids, 2 * rw, get), 2 * out, rtol=1e-13)
    one = O.moe_forward(x[1:2], np.array([[3]]), np.array([[rw[1, 0] + rw[1, 1]]]), get)
    assert np.allclose(out[1], one[0], rtol=1e-12)
    # j order and token subsets do not change a row
    assert np.allclose(O.moe_forward(x, ids[:, ::-1], rw[:, ::-1], get), out, rtol=1e-12)
    assert np.allclose(O.moe_forward(x, ids, rw, get, tokens=[2])[0], out[2], rtol=1e-13)


def test_expert_relabelling_leaves_output_unchanged():
    get = _experts()
    x = np.random.default_rng(4).standard_normal((5, H))
    ids = np.random.default_rng(5).integers(0, E, size=(5, 3))
    rw = np.random.default_rng(6).uniform(size=(5, 3))
    perm = np.array([2, 0, 3, 1])
    inv = np.argsort(perm)
    a = O.moe_forward(x, ids, rw, get)
    b = O.moe_forward(x, perm[ids], rw, lambda e, p: get(inv[e], p))
    assert np.allclose(a, b, rtol=1e-13)


# ---------------------------------------------------------------- additive
def test_zero_scale_stage_is_the_base_exactly():
    get = _experts(cbs=(CB_MCG,) * 4, Ks=(3,) * 4)
    x = np.random.default_rng(7).standard_normal((3, H))
    ids = np.array([[0, 1], [2, 3], [1, 1]])
    rw = np.full((3, 2), 0.5)
    res_T = {k: make_projection([99, *k], get(*k).in_features, get(*k).out_features, 2,
                                CB_MCG).trellis
             for k in [(e, p) for e in range(E) for p in range(3)]}
    base = O.moe_forward(x, ids, rw, get)
    zero = O.moe_forward(x, ids, rw, get, get_residuals=lambda e, p: [(0.0, res_T[e, p], 2)])
    assert np.array_equal(base, zero)


def test_residual_with_base_codes_and_unit_scale_doubles_the_weights():
    p = make_projection([13], 256, 128, 3, CB_MCG)
    x = np.random.default_rng(8).standard_normal((4, 256))
    y2 = O.linear(x, p, residuals=[(1.0, p.trellis, 3)])
    q = make_projection([13], 256, 128, 3, CB_MCG)
    q.scale = (q.scale.astype(np.float64) * 2).astype(np.float16)
    assert np.allclose(y2, O.linear(x, q), rtol=1e-12)
    y3 = O.linear(x, p, residuals=[(0.25, p.trellis, 3), (0.5, p.trellis, 3)])
    assert np.allclose(y3, 1.75 * O.linear(x, p), rtol=1e-12)


@pytest.mark.parametrize("base_cb", [CB_MCG, CB_3INST, CB_MUL1])
def test_residual_is_an_mcg_projection_with_the_base_rotations(base_cb):
    # a stage adds alpha times the mcg projection of its own codes and width
    # under the base's suh, svh and scale: the sum of two plain linears, each
    # pinned on its own above
    from workloads import Projection
    p = make_projection([21, base_cb], 256, 384, 4, base_cb)
    t2 = make_projection([22], 256, 384, 2, CB_MCG).trellis
    t5 = make_projection([23], 256, 384, 5, CB_MCG).trellis
    x = np.random.default_rng(24).standard_normal((5, 256))

    def with_codes(trellis, K):
        return Projection(trellis, p.suh, p.svh, p.scale, K, CB_MCG)

    got = O.linear(x, p, residuals=[(0.3, t2, 2), (-0.125, t5, 5)])
    want = (O.linear(x, p) + 0.3 * O.linear(x, with_codes(t2, 2))
            - 0.125 * O.linear(x, with_codes(t5, 5)))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
