"""Pins for the FP64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: hand-derived closed
forms (tests/golden/closed_forms.json), brute-force enumeration of every top-k
subset, library routines (scipy softmax, numpy stable argsort, numpy float16
rounding, numpy matmul) and invariants of the dispatch.  The cases are chosen
so that a dropped term, a wrong sign, a swapped gate/up, a transposed weight or
a wrong tie rule fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
_ENV = {"log": math.log, "exp": math.exp, "inf": math.inf, "nan": math.nan}


def _val(v):
    return float(eval(v, {"__builtins__": {}}, _ENV)) if isinstance(v, str) else float(v)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden()["routing"], ids=lambda c: c["name"])
def test_route_closed_forms(oracle_mod, case):
    logits = _f32([[_val(v) for v in case["logits"]]])
    # logits given as exact expressions; rounding them to f32 moves the softmax
    # by <= 2^-24 relative, far inside the 1e-6 comparison below
    idx, w_pre, w_cast = oracle_mod.route(logits, "f32", case["top_k"], case["renormalize"])
    assert idx[0].tolist() == case["idx"]
    want = np.array([_val(v) for v in case["weights"]])
    got = w_pre[0]
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_allclose(got[ok], want[ok], rtol=1e-6, atol=1e-12)


def _brute_force_topk(row, k):
    """The unique k-subset whose members all beat every non-member by
    (larger logit, then lower id); found by enumerating all subsets."""
    E = len(row)

    def beats(a, b):
        return row[a] > row[b] or (row[a] == row[b] and a < b)

    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(beats(a, b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    S = winners[0]
    # slot order: descending weight, ties to the lower id
    return sorted(S, key=lambda e: (-row[e], e))


def test_route_brute_force_with_frequent_ties(oracle_mod):
    rng = np.random.default_rng(1234)
    values = np.array([-np.inf, -2.0, -0.0, 0.0, 0.5, 0.5, 1.0, 3.0])
    for _ in range(400):
        E = int(rng.integers(1, 8))
        k = int(rng.integers(1, E + 1))
        row = rng.choice(values, size=E)
        if np.all(row == -np.inf):
            row[0] = 0.0
        idx, w_pre, _ = oracle_mod.route(_f32([row]), "f32", k, False)
        assert idx[0].tolist() == _brute_force_topk(list(row), k)
        # weights are the softmax at the selected ids
        ex = np.exp(row - row.max())
        p = ex / ex.sum()
        np.testing.assert_allclose(w_pre[0], p[idx[0]], rtol=1e-14, atol=1e-300)


def test_route_matches_scipy_softmax(oracle_mod):
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    logits = _f32(rng.normal(size=(64, 37)) * 3)
    ld = logits.astype(np.float64)
    p = scipy_special.softmax(ld, axis=1)
    for k in (1, 5, 37):
        idx, w_pre, _ = oracle_mod.route(logits, "f32", k, False)
        np.testing.assert_allclose(w_pre, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=1e-13)
        # selected ids are the k largest logits, in descending order
        order = np.argsort(-ld, axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, order)
    # k = E with renormalisation reproduces the whole softmax (permuted)
    idx, w_pre, _ = oracle_mod.route(logits, "f32", 37, True)
    np.testing.assert_allclose(w_pre, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=1e-13)


def test_route_renormalised_weights_sum_to_one(oracle_mod):
    rng = np.random.default_rng(3)
    logits = _f32(rng.normal(size=(200, 64)))
    for k in (1, 2, 6, 64):
        _, w_pre, _ = oracle_mod.route(logits, "f32", k, True)
        np.testing.assert_allclose(w_pre.sum(1), 1.0, rtol=0, atol=1e-15 * k)
        if k == 1:
            assert np.all(w_pre == 1.0)


def test_route_single_expert_and_uniform(oracle_mod):
    idx, w_pre, _ = oracle_mod.route(_f32([[0.7], [-3.0]]), "f32", 1, False)
    assert idx.ravel().tolist() == [0, 0] and np.all(w_pre == 1.0)
    E = 16
    idx, w_pre, _ = oracle_mod.route(_f32(np.zeros((3, E))), "f32", 4, False)
    assert np.all(idx == np.arange(4)) and np.allclose(w_pre, 1.0 / E, rtol=1e-15)


def test_route_nan_rule(oracle_mod):
    rows = [
        [0.0, np.nan, 1.0, 2.0],
        [0.0, np.inf, 1.0, 2.0],
        [-np.inf] * 4,
        [np.nan] * 4,
        [-np.inf, 1.0, -np.inf, 0.0],   # some -inf: finite
        [np.inf, -np.inf, np.nan, 0.0],
    ]
    idx, w_pre, w_cast = oracle_mod.route(_f32(rows), "f32", 3, True)
    for t in (0, 1, 2, 3, 5):
        assert idx[t].tolist() == [0, 1, 2]
        assert np.all(np.isnan(w_pre[t])) and np.all(np.isnan(w_cast[t]))
    assert idx[4].tolist() == [1, 3, 0]
    assert np.all(np.isfinite(w_pre[4]))
    np.testing.assert_allclose(w_pre[4], [math.e / (math.e + 1), 1 / (math.e + 1), 0.0], rtol=1e-15)


def test_route_cast_uses_logits_dtype(oracle_mod):
    """Stored weights are the FP64 weights rounded to the logits dtype."""
    rng = np.random.default_rng(11)
    logits = rng.normal(size=(50, 9)).astype(np.float16)
    idx, w_pre, w_cast = oracle_mod.route(logits, "f16", 3, True)
    np.testing.assert_array_equal(w_cast, w_pre.astype(np.float16).astype(np.float64))


# --------------------------------------------------------------------------
# exact decoding and RNE rounding of the storage formats
# --------------------------------------------------------------------------

def test_decode_every_f16_and_bf16_pattern(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle_mod.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(f16), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(f16[ok], ref[ok])
    assert np.array_equal(np.signbit(f16[ok]), np.signbit(ref[ok]))
    bf = oracle_mod.decode(bits, "bf16")
    with np.errstate(invalid="ignore"):  # the NaN patterns widen to NaN
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(np.isnan(bf), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(bf[ok], ref[ok])


def test_round_to_f16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.normal(size=3000) * 10.0 ** rng.integers(-9, 6, size=3000),
                           [65519.0, 65520.0, 65504.0, 1e-8, 2.0 ** -25, 3 * 2.0 ** -26, -0.0]])
    for v in vals:
        with np.errstate(over="ignore"):  # values past the f16 range round to infinity
            want = float(np.float16(v))
        assert oracle_mod.round_to_dtype(v, "f16") == want, v
        assert oracle_mod.round_to_dtype(v, "f32") == float(np.float32(v)), v


def test_round_to_bf16_is_nearest_even(oracle_mod):
    """Brute force: the result is a bf16 value, no bf16 value is closer, and a
    tie goes to the even mantissa."""
    rng = np.random.default_rng(9)
    vals = np.concatenate([rng.normal(size=2000) * 10.0 ** rng.integers(-30, 30, size=2000),
                           [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40]])
    for v in vals:
        r = oracle_mod.round_to_dtype(v, "bf16")
        rb = np.array([r], np.float32).view(np.uint32)[0]
        assert rb & 0xFFFF == 0 and float(np.float32(r)) == r
        # neighbours of r in bf16
        up = (np.array([rb + 0x10000], np.uint32).view(np.float32)[0]).astype(np.float64)
        dn = (np.array([rb - 0x10000], np.uint32).view(np.float32)[0]).astype(np.float64)
        for nb in (up, dn):
            if np.isfinite(nb) and np.sign(nb) == np.sign(r):
                assert abs(v - r) <= abs(v - nb)
                if abs(v - r) == abs(v - nb):
                    assert (rb >> 16) & 1 == 0


# --------------------------------------------------------------------------
# dispatch
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden()["dispatch"], ids=lambda c: c["name"])
def test_dispatch_closed_forms(oracle_mod, case):
    idx = np.array(case["idx"], np.uint32)
    offsets, row_experts, perm, bad = oracle_mod.dispatch(idx, case["E"])
    assert bad == 0
    assert offsets.tolist() == case["offsets"]
    assert perm.tolist() == case["perm"]
    assert row_experts.tolist() == case["row_experts"]


def test_dispatch_invariants_and_stable_sort(oracle_mod):
    rng = np.random.default_rng(2)
    for T, E, k in [(1, 1, 1), (37, 5, 3), (300, 64, 6), (128, 8, 8), (0, 4, 2)]:
        logits = _f32(rng.normal(size=(T, E)))
        idx, _, _ = oracle_mod.route(logits, "f32", k, False)
        offsets, row_experts, perm, bad = oracle_mod.dispatch(idx, E)
        n = T * k
        assert bad == 0 and offsets[0] == 0 and offsets[-1] == n
        assert np.all(np.diff(offsets.astype(np.int64)) >= 0)
        assert sorted(perm.tolist()) == list(range(n))
        # every token appears exactly k times
        assert np.array_equal(np.bincount(perm // k, minlength=T), np.full(T, k))
        flat = idx.ravel()
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(row_experts, flat[perm])
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(np.diff(seg.astype(np.int64)) > 0)   # ascending token order
            assert np.all(flat[seg] == e)


def test_dispatch_duplicates_and_invalid(oracle_mod):
    idx = np.array([[2, 2], [7, 0], [0, 2]], np.uint32)   # duplicate expert in row 0, id 7 >= E
    offsets, row_experts, perm, bad = oracle_mod.dispatch(idx, 3)
    assert bad == 1
    assert offsets.tolist() == [0, 2, 2, 5]
    assert perm.tolist() == [3, 4, 0, 1, 5, 0xFFFFFFFF]
    assert np.array_equal(perm[:5], np.argsort(np.where(idx.ravel() < 3, idx.ravel(), 99),
                                               kind="stable")[:5])


# --------------------------------------------------------------------------
# experts and combine
# --------------------------------------------------------------------------

def _silu(z):
    return z / (1.0 + np.exp(-z))


def _dense_masked_forward(x, logits, gate, up, down, k, renorm):
    """Independent evaluation: loop over ALL experts with a selection mask,
    no dispatch at all.  Routing weights via scipy's softmax and a stable
    argsort on (-logit), cast to f32 (the stored dtype of these cases)."""
    from scipy.special import softmax
    T, E = logits.shape
    p = softmax(logits, axis=1)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    w = np.take_along_axis(p, order, 1)
    if renorm:
        w = w / w.sum(1, keepdims=True)
    w = w.astype(np.float32).astype(np.float64)
    y = np.zeros((T, gate.shape[2]))
    for e in range(E):
        a = _silu(x @ gate[e].T) * (x @ up[e].T)       # [T, I]
        o = a @ down[e].T                               # [T, H]
        sel = (order == e)                              # [T, k]
        coef = (w * sel).sum(1)                         # weight of e for each token (0 if unselected)
        y += coef[:, None] * o
    return y, order


@pytest.mark.parametrize("T,E,k,H,I,renorm", [(23, 4, 2, 8, 12, True), (40, 7, 3, 16, 6, False),
                                                (9, 5, 5, 5, 9, True)])
def test_chain_equals_dense_masked_forward(oracle_mod, T, E, k, H, I, renorm):
    pytest.importorskip("scipy")
    rng = np.random.default_rng(T * 100 + E)
    x = _f32(rng.normal(size=(T, H)))
    logits = _f32(rng.normal(size=(T, E)))
    gate = _f32(rng.normal(size=(E, I, H)) / np.sqrt(H))
    up = _f32(rng.normal(size=(E, I, H)) / np.sqrt(H))
    down = _f32(rng.normal(size=(E, H, I)) / np.sqrt(I))
    y_ref, order = _dense_masked_forward(x.astype(np.float64), logits.astype(np.float64),
                                         gate.astype(np.float64), up.astype(np.float64),
                                         down.astype(np.float64), k, renorm)
    # staged chain: route -> dispatch -> experts -> combine
    idx, w_pre, w_cast = oracle_mod.route(logits, "f32", k, renorm)
    assert np.array_equal(idx, order)
    offsets, row_experts, perm, _ = oracle_mod.dispatch(idx, E)
    x_disp = x.astype(np.float64)[perm // k]
    eo = oracle_mod.experts(x_disp, offsets, gate, up, down, "f32")
    y = oracle_mod.combine(eo, perm, w_cast)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    # per-token forward on a sample
    toks = [0, T // 2, T - 1]
    idx_s, _, y_s = oracle_mod.forward_tokens(x, logits, gate, up, down, "f32", "f32", k, renorm, toks)
    assert np.array_equal(idx_s, idx[toks])
    np.testing.assert_allclose(y_s, y_ref[toks], rtol=1e-12, atol=1e-12)


def test_single_expert_is_plain_swiglu_mlp(oracle_mod):
    """E=1, k=1, renormalised: y = W_down (silu(W_gate x) * (W_up x))."""
    rng = np.random.default_rng(4)
    T, H, I = 13, 24, 40
    x = _f32(rng.normal(size=(T, H)))
    gate = _f32(rng.normal(size=(1, I, H)) / 5)
    up = _f32(rng.normal(size=(1, I, H)) / 5)
    down = _f32(rng.normal(size=(1, H, I)) / 6)
    logits = _f32(rng.normal(size=(T, 1)))
    xd = x.astype(np.float64)
    ref = (_silu(xd @ gate[0].T.astype(np.float64)) * (xd @ up[0].T.astype(np.float64))) \
        @ down[0].T.astype(np.float64)
    idx, w_pre, w_cast = oracle_mod.route(logits, "f32", 1, True)
    assert np.all(w_cast == 1.0)
    offsets, _, perm, _ = oracle_mod.dispatch(idx, 1)
    eo = oracle_mod.experts(xd[perm], offsets, gate, up, down, "f32")
    y = oracle_mod.combine(eo, perm, w_cast)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("case", _golden()["experts"], ids=lambda c: c["name"])
def test_expert_closed_forms(oracle_mod, case):
    E, H, I = case["E"], case["H"], case["I"]
    x = _f32(np.reshape(case["x"], (1, H)))
    gate = _f32(np.reshape(case["gate"], (E, I, H)))
    up = _f32(np.reshape(case["up"], (E, I, H)))
    down = _f32(np.reshape(case["down"], (E, H, I)))
    logits = _f32(np.zeros((1, E)))
    want = np.array([_val(v) for v in np.atleast_1d(case["y"])])
    _, _, y = oracle_mod.forward_tokens(x, logits, gate, up, down, "f32", "f32", case["top_k"], True, [0])
    np.testing.assert_allclose(y[0], want, rtol=1e-15, atol=1e-15)


def test_combine_poisoned_and_undispatched_rows_are_nan(oracle_mod):
    eo = np.arange(12, dtype=np.float64).reshape(6, 2)
    perm = np.array([1, 2, 0, 4, 3, 0xFFFFFFFF], np.uint32)
    w = np.array([[0.5, 0.25], [np.nan, np.nan], [1.0, 1.0]])
    y = oracle_mod.combine(eo, perm, w)
    # token 0: slot 0 -> row 2, slot 1 -> row 0
    np.testing.assert_array_equal(y[0], 0.5 * eo[2] + 0.25 * eo[0])
    assert np.all(np.isnan(y[1]))          # NaN weights
    assert np.all(np.isnan(y[2]))          # slot 5 never dispatched
