"""Pins for the oracle's sigmoid group-limited routing (CPU only).

User guide section 10: sigmoid scores, an FP32 correction bias that only
affects selection, `selected_groups` best groups by max (or top-two sum) of
corrected scores, then top_k experts inside them; ties to lower ids; weights
are the original sigmoid values, optionally renormalised, times scale."""
import itertools

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))


def _brute_force(c, groups, sel, k, top_two):
    """Exhaustive reference on FP32 corrected scores c [E]."""
    E = len(c)
    gs = E // groups

    def gscore(g):
        v = sorted(c[g * gs:(g + 1) * gs], reverse=True)
        return np.float32(v[0] + v[1]) if top_two else v[0]

    gsc = [gscore(g) for g in range(groups)]

    def beats(va, a, vb, b):
        return va > vb or (va == vb and a < b)

    winners = [S for S in itertools.combinations(range(groups), sel)
               if all(beats(gsc[a], a, gsc[b], b) for a in S for b in range(groups) if b not in S)]
    assert len(winners) == 1
    allowed = [e for e in range(E) if e // gs in winners[0]]
    exp_w = [S for S in itertools.combinations(allowed, k)
             if all(beats(c[a], a, c[b], b) for a in S for b in allowed if b not in S)]
    assert len(exp_w) == 1
    return sorted(exp_w[0], key=lambda e: (-c[e], e))


def test_selection_matches_exhaustive_search(oracle_mod):
    rng = np.random.default_rng(10)
    for _ in range(300):
        groups = int(rng.choice([1, 2, 3, 4]))
        gs = int(rng.integers(1, 4)) if groups > 1 else int(rng.integers(1, 7))
        E = groups * gs
        top_two = bool(rng.integers(0, 2)) and gs >= 2
        sel = int(rng.integers(1, groups + 1))
        k = int(rng.integers(1, sel * gs + 1))
        logits = _f32(rng.choice([-2.0, -0.5, 0.0, 0.0, 1.0, 3.0], size=(1, E)))
        bias = _f32(rng.choice([0.0, 0.0, 0.25, -0.25, 0.5], size=E))
        idx, w_pre, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", k, groups, sel, top_two,
                                                         False, 1.0, bias)
        # corrected scores in FP32: library sigmoid rounded once, FP32 add
        c = (scipy_special.expit(logits[0].astype(np.float64)).astype(np.float32) + bias).astype(np.float32)
        assert idx[0].tolist() == _brute_force(list(c), groups, sel, k, top_two)
        np.testing.assert_allclose(w_pre[0], scipy_special.expit(logits[0].astype(np.float64))[idx[0]],
                                   rtol=1e-15)


def test_single_group_without_bias_is_plain_topk(oracle_mod):
    rng = np.random.default_rng(11)
    logits = _f32(rng.normal(size=(50, 48)))
    for k, renorm, scale in [(1, True, 1.0), (6, False, 2.5), (48, True, 0.5)]:
        idx, w_pre, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", k, 1, 1, False, renorm, scale)
        order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, order)
        s = np.take_along_axis(scipy_special.expit(logits.astype(np.float64)), order, 1)
        if renorm:
            s = s / s.sum(1, keepdims=True)
        np.testing.assert_allclose(w_pre, s * scale, rtol=1e-14)


def test_all_groups_kept_equals_topk_by_corrected_score(oracle_mod):
    rng = np.random.default_rng(12)
    logits = _f32(rng.normal(size=(40, 32)))
    bias = _f32(rng.normal(size=32) * 0.3)
    idx, _, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", 5, 8, 8, True, True, 1.0, bias)
    c = (scipy_special.expit(logits.astype(np.float64)).astype(np.float32) + bias).astype(np.float32)
    order = np.argsort(-c.astype(np.float64), axis=1, kind="stable")[:, :5]
    assert np.array_equal(idx, order)


def test_bias_moves_selection_not_weights(oracle_mod):
    logits = _f32([[2.0, 1.0, 0.0, -1.0]])
    bias = _f32([0.0, 0.0, 0.0, 5.0])
    idx, w_pre, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", 1, 1, 1, False, False, 1.0, bias)
    assert idx[0].tolist() == [3]
    assert w_pre[0, 0] == pytest.approx(1.0 / (1.0 + np.e), rel=1e-15)


def test_top_two_group_score_closed_form(oracle_mod):
    # logits 0 give sigmoid 1/2; the bias sets corrected scores exactly to
    # [0.875, 0.125 | 0.625, 0.625]: max picks group 0, top-two sum picks group 1
    logits = _f32([[0.0, 0.0, 0.0, 0.0]])
    bias = _f32([0.375, -0.375, 0.125, 0.125])
    idx, w, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", 2, 2, 1, False, True, 2.5, bias)
    assert idx[0].tolist() == [0, 1]
    idx, w, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", 2, 2, 1, True, True, 2.5, bias)
    assert idx[0].tolist() == [2, 3]
    np.testing.assert_allclose(w[0], [1.25, 1.25], rtol=1e-15)   # 0.5/(0.5+0.5) * 2.5


def test_nan_rows(oracle_mod):
    logits = _f32([[0.0, np.nan, 1.0, 2.0], [0.0, 1.0, np.inf, -np.inf]])
    idx, w, wc = oracle_mod.route_sigmoid_grouped(logits, "f32", 2, 2, 1, False, True, 1.0)
    assert idx[0].tolist() == [0, 1] and np.isnan(w[0]).all() and np.isnan(wc[0]).all()
    # +-inf are ordinary for a sigmoid: 1 and 0
    # group scores max(0.5, 0.731) < max(1, 0): group 1 is kept
    assert idx[1].tolist() == [2, 3]
    assert np.all(np.isfinite(w[1]))
