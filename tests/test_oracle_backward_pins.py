"""Pins for the oracle's first-order training backward (CPU only).

Every gradient is checked against central finite differences of the oracle's
own FP64 forward functions (an independent derivation: a wrong sign, a
dropped term or a transposed index in a backward formula fails), and the
selected router weights against the routers' own weights."""
import numpy as np
import pytest

EPS = 2.0 ** -10   # perturbation; weights below live on a 2^-8 grid so w +- EPS is exact in f32


def _grid_f32(rng, shape, scale):
    """Random values on a 2^-8 grid (exact in f32, and so is v +- 2^-10)."""
    return np.ascontiguousarray((np.round(rng.normal(size=shape) * scale * 256) / 256).astype(np.float32))


def _setup(rng, T=7, E=3, k=2, H=5, I=4):
    x = rng.normal(size=(T, H))
    logits = rng.normal(size=(T, E)).astype(np.float32)
    gate = _grid_f32(rng, (E, I, H), 0.5)
    up = _grid_f32(rng, (E, I, H), 0.5)
    down = _grid_f32(rng, (E, H, I), 0.5)
    return x, logits, gate, up, down


def test_expert_gradients_match_finite_differences(oracle_mod):
    rng = np.random.default_rng(21)
    T, E, k, H, I = 7, 3, 2, 5, 4
    x, logits, gate, up, down = _setup(rng, T, E, k, H, I)
    idx, _, _ = oracle_mod.route(logits, "f32", k, True)
    off, _, perm, _ = oracle_mod.dispatch(idx, E)
    xd = x[perm // k]
    dout = rng.normal(size=(T * k, H))

    def loss(xd_, g_, u_, d_):
        return float((oracle_mod.experts(xd_, off, g_, u_, d_, "f32") * dout).sum())

    dinput, dgate, dup, ddown = oracle_mod.experts_backward(xd, off, gate, up, down, "f32", dout)
    # input rows
    for r in range(T * k):
        for h in range(H):
            p, m = xd.copy(), xd.copy()
            p[r, h] += 1e-5
            m[r, h] -= 1e-5
            fd = (loss(p, gate, up, down) - loss(m, gate, up, down)) / 2e-5
            assert dinput[r, h] == pytest.approx(fd, rel=1e-6, abs=1e-8)
    # weights (exact perturbations on the 2^-8 grid)
    for name, W, G in (("gate", gate, dgate), ("up", up, dup), ("down", down, ddown)):
        for pos in np.ndindex(W.shape):
            p, m = W.copy(), W.copy()
            p[pos] += np.float32(EPS)
            m[pos] -= np.float32(EPS)
            args_p = {"gate": gate, "up": up, "down": down, name: p}
            args_m = {"gate": gate, "up": up, "down": down, name: m}
            fd = (loss(xd, args_p["gate"], args_p["up"], args_p["down"])
                  - loss(xd, args_m["gate"], args_m["up"], args_m["down"])) / (2 * EPS)
            assert G[pos] == pytest.approx(fd, rel=1e-4, abs=1e-6), (name, pos)


def test_expert_gradients_of_unused_experts_are_zero(oracle_mod):
    rng = np.random.default_rng(22)
    x, logits, gate, up, down = _setup(rng, 6, 4, 1, 5, 3)
    logits[:, 3] = -50.0        # expert 3 never selected
    idx, _, _ = oracle_mod.route(logits, "f32", 1, True)
    off, _, perm, _ = oracle_mod.dispatch(idx, 4)
    _, dg, du, dd = oracle_mod.experts_backward(x[perm], off, gate, up, down, "f32",
                                                rng.normal(size=(6, 5)))
    assert np.all(dg[3] == 0) and np.all(du[3] == 0) and np.all(dd[3] == 0)


def test_combine_gradients_match_finite_differences(oracle_mod):
    rng = np.random.default_rng(23)
    T, E, k, H = 6, 4, 3, 5
    logits = rng.normal(size=(T, E)).astype(np.float32)
    idx, _, w_cast = oracle_mod.route(logits, "f32", k, True)
    off, _, perm, _ = oracle_mod.dispatch(idx, E)
    eo = rng.normal(size=(T * k, H))
    dy = rng.normal(size=(T, H))
    dex, dw = oracle_mod.combine_backward(eo, perm, w_cast, dy)

    def loss(eo_, w_):
        return float((oracle_mod.combine(eo_, perm, w_) * dy).sum())

    for r in range(T * k):
        for h in range(H):
            p, m = eo.copy(), eo.copy()
            p[r, h] += 1e-4
            m[r, h] -= 1e-4
            assert dex[r, h] == pytest.approx((loss(p, w_cast) - loss(m, w_cast)) / 2e-4, rel=1e-8, abs=1e-10)
    for t in range(T):
        for j in range(k):
            p, m = w_cast.copy(), w_cast.copy()
            p[t, j] += 1e-4
            m[t, j] -= 1e-4
            assert dw[t, j] == pytest.approx((loss(eo, p) - loss(eo, m)) / 2e-4, rel=1e-8, abs=1e-10)


def test_dispatch_backward_is_the_gather_transpose(oracle_mod):
    rng = np.random.default_rng(24)
    T, E, k, H = 9, 5, 3, 4
    idx, _, _ = oracle_mod.route(rng.normal(size=(T, E)).astype(np.float32), "f32", k, False)
    _, _, perm, _ = oracle_mod.dispatch(idx, E)
    dinput = rng.normal(size=(T * k, H))
    dx = oracle_mod.dispatch_backward(dinput, perm, T, k)
    x = rng.normal(size=(T, H))
    # <dinput, gather(x)> == <dispatch_backward(dinput), x> for every x
    assert (dinput * x[perm // k]).sum() == pytest.approx((dx * x).sum(), rel=1e-13)
    # each token receives exactly its k rows
    for t in range(T):
        np.testing.assert_allclose(dx[t], dinput[np.where(perm // k == t)[0]].sum(0), rtol=1e-14)


@pytest.mark.parametrize("scoring,renorm,scale", [("softmax", False, 1.0), ("softmax", True, 1.0),
                                                  ("softmax", True, 2.5), ("sigmoid", False, 1.0),
                                                  ("sigmoid", True, 1.5)])
def test_router_gradients_match_finite_differences(oracle_mod, scoring, renorm, scale):
    rng = np.random.default_rng(25)
    T, E, k = 5, 6, 3
    logits = rng.normal(size=(T, E))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    idx[1, 2] = idx[1, 0]            # repeated index: gather semantics
    dw = rng.normal(size=(T, k))
    dl = oracle_mod.router_backward(logits, idx, dw, scoring, renorm, scale)

    def loss(l_):
        return float((oracle_mod.selected_router_weights(l_, idx, scoring, renorm, scale) * dw).sum())

    for t in range(T):
        for e in range(E):
            p, m = logits.copy(), logits.copy()
            p[t, e] += 1e-5
            m[t, e] -= 1e-5
            assert dl[t, e] == pytest.approx((loss(p) - loss(m)) / 2e-5, rel=1e-6, abs=1e-9)


def test_selected_router_weights_equal_the_routers(oracle_mod):
    rng = np.random.default_rng(26)
    logits = rng.normal(size=(30, 16)).astype(np.float32)
    idx, w_pre, _ = oracle_mod.route(logits, "f32", 4, True)
    w = oracle_mod.selected_router_weights(logits.astype(np.float64), idx.astype(np.int64), "softmax", True)
    np.testing.assert_allclose(w, w_pre, rtol=1e-14)
    idx, w_pre, _ = oracle_mod.route_sigmoid_grouped(logits, "f32", 4, 1, 1, False, True, 2.0)
    w = oracle_mod.selected_router_weights(logits.astype(np.float64), idx.astype(np.int64), "sigmoid", True, 2.0)
    np.testing.assert_allclose(w, w_pre, rtol=1e-14)


def test_invalid_router_indices_give_nan_rows(oracle_mod):
    logits = np.zeros((3, 4))
    idx = np.array([[0, 1], [2, 7], [3, -1]])
    dl = oracle_mod.router_backward(logits, idx, np.ones((3, 2)), "softmax", True)
    assert np.all(np.isfinite(dl[0])) and np.all(np.isnan(dl[1])) and np.all(np.isnan(dl[2]))
    w = oracle_mod.selected_router_weights(logits, idx, "sigmoid", False)
    assert np.all(np.isfinite(w[0])) and np.all(np.isnan(w[1:]))
