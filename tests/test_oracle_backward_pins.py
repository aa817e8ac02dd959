"""Pins of the oracle's backward pass (reverse mode of the scan, slots held fixed) against
things other than itself:
  * central finite differences of the forward oracle (itself pinned in test_oracle_pins.py)
    for every gradient: v, alpha, beta, the selected write and read scores, M_0;
  * an exact identity: with alpha, beta and the scores fixed, o and M_T are linear in
    (v, M_0) jointly and vanish at (0, 0), so L(v, M_0) = <dL/dv, v> + <dL/dM_0, M_0> for
    L = sum_t <dO_t, o_t> + <dM_T, M_T> ("Meccanismo Core" items 3 and 4: the delta update
    is affine in the old row and in v, the read is linear in the table);
  * the half-entry gradients of the scores (a selected score is half0[i] + half1[j],
    "Meccanismo Core" item 2) against finite differences of the whole forward, selection
    included, where the perturbation leaves the selection unchanged.
"""
import numpy as np
import pytest

import oracle


def _problem(seed, nh=2, T=7, S=4, dv=3, W=3, R=4):
    rng = np.random.default_rng(seed)
    kp = rng.standard_normal((nh, T, 2, S)).astype(np.float32)
    qp = rng.standard_normal((nh, T, 2, S)).astype(np.float32)
    iw, sw = oracle.select(kp, W)
    ir, sr = oracle.select(qp, R)
    return dict(kp=kp, qp=qp, iw=iw, sw=sw, ir=ir, sr=sr,
                v=rng.standard_normal((nh, T, dv)).astype(np.float32),
                alpha=rng.uniform(0.8, 1.0, (nh, T)).astype(np.float32),
                beta=rng.uniform(0.2, 1.0, (nh, T)).astype(np.float32),
                M0=0.5 * rng.standard_normal((nh, S * S, dv)),
                dO=rng.standard_normal((nh, T, dv)),
                dMT=rng.standard_normal((nh, S * S, dv)), W=W, R=R, S=S)


def _loss(p, **over):
    q = dict(p, **over)
    M = np.array(q["M0"], np.float64, order="C", copy=True)
    o = oracle.scan(M, q["iw"], q["sw"], q["ir"], q["sr"], q["v"], q["alpha"], q["beta"])
    return float(np.sum(q["dO"] * o) + np.sum(q["dMT"] * M))


def _grads(p):
    return oracle.scan_backward(p["M0"], p["iw"], p["sw"], p["ir"], p["sr"], p["v"], p["alpha"], p["beta"],
                                p["dO"], p["dMT"])


def _fd32(p, name, index, h=2.0 ** -9):
    """Central difference in an fp32 input, divided by the perturbation actually applied."""
    x = p[name]
    up, dn = x.copy(), x.copy()
    up[index] = np.float32(x[index] + np.float32(h))
    dn[index] = np.float32(x[index] - np.float32(h))
    return (_loss(p, **{name: up}) - _loss(p, **{name: dn})) / (float(up[index]) - float(dn[index]))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_backward_matches_finite_differences(seed):
    p = _problem(seed)
    g = _grads(p)
    rng = np.random.default_rng(100 + seed)
    nh, T, dv = p["v"].shape
    checks = 0
    for _ in range(6):
        h, t, c = rng.integers(nh), rng.integers(T), rng.integers(dv)
        assert _fd32(p, "v", (h, t, c)) == pytest.approx(g["dv"][h, t, c], rel=2e-4, abs=2e-5)
        assert _fd32(p, "alpha", (h, t)) == pytest.approx(g["dalpha"][h, t], rel=2e-4, abs=2e-5)
        assert _fd32(p, "beta", (h, t)) == pytest.approx(g["dbeta"][h, t], rel=2e-4, abs=2e-5)
        i, j = rng.integers(p["W"]), rng.integers(p["R"])
        assert _fd32(p, "sw", (h, t, i)) == pytest.approx(g["dsc_w"][h, t, i], rel=2e-4, abs=2e-5)
        assert _fd32(p, "sr", (h, t, j)) == pytest.approx(g["dsc_r"][h, t, j], rel=2e-4, abs=2e-5)
        n = rng.integers(p["M0"].shape[1])
        up, dn = p["M0"].copy(), p["M0"].copy()
        up[h, n, c] += 1e-6
        dn[h, n, c] -= 1e-6
        fd = (_loss(p, M0=up) - _loss(p, M0=dn)) / 2e-6
        assert fd == pytest.approx(g["dM0"][h, n, c], rel=1e-6, abs=1e-8)
        checks += 6
    assert checks == 36


@pytest.mark.parametrize("seed", [3, 4])
def test_loss_is_the_inner_product_of_the_linear_gradients(seed):
    p = _problem(seed, T=9, S=5, dv=4, W=6, R=7)
    g = _grads(p)
    L = _loss(p)
    lin = float(np.sum(g["dv"] * p["v"].astype(np.float64)) + np.sum(g["dM0"] * p["M0"]))
    assert lin == pytest.approx(L, rel=1e-12, abs=1e-12)
    # and the zero point is zero
    assert _loss(p, v=np.zeros_like(p["v"]), M0=np.zeros_like(p["M0"])) == 0.0


def test_untouched_rows_pass_their_gradient_through():
    """A slot that is never written keeps M_0's value, so dL/dM_0 there is dM_T plus the
    reads' weights times dO."""
    p = _problem(5)
    g = _grads(p)
    nh, T, _ = p["v"].shape
    for h in range(nh):
        written = set(p["iw"][h].ravel().tolist())
        for n in range(p["M0"].shape[1]):
            if n in written:
                continue
            want = p["dMT"][h, n].copy()
            for t in range(T):
                e = np.exp(p["sr"][h, t].astype(np.float64) - p["sr"][h, t].max())
                r = e / e.sum()
                for j in np.nonzero(p["ir"][h, t] == n)[0]:
                    want += r[j] * p["dO"][h, t]
            assert np.allclose(g["dM0"][h, n], want, rtol=1e-12, atol=1e-12)


def test_half_entry_gradients_through_the_selection():
    p = _problem(6, T=5)
    g = _grads(p)
    dkp = oracle.select_backward(p["S"], p["iw"], g["dsc_w"])
    dqp = oracle.select_backward(p["S"], p["ir"], g["dsc_r"])

    def full_loss(kp, qp):
        r = oracle.forward(kp, qp, p["v"], p["alpha"], p["beta"], p["M0"], p["W"], p["R"])
        L = float(np.sum(p["dO"] * r["o"]) + np.sum(p["dMT"] * r["M"]))
        return L, r["idx_w"], r["idx_r"]

    rng = np.random.default_rng(7)
    checked = 0
    for _ in range(40):
        which = rng.integers(2)
        x = (p["kp"], p["qp"])[which]
        ix = (0, rng.integers(x.shape[1]), rng.integers(2), rng.integers(p["S"]))
        hh = np.float32(2.0 ** -11)
        up, dn = x.copy(), x.copy()
        up[ix] += hh
        dn[ix] -= hh
        args_up = (up, p["qp"]) if which == 0 else (p["kp"], up)
        args_dn = (dn, p["qp"]) if which == 0 else (p["kp"], dn)
        Lu, iwu, iru = full_loss(*args_up)
        Ld, iwd, ird = full_loss(*args_dn)
        if not (np.array_equal(iwu, p["iw"]) and np.array_equal(iwd, p["iw"]) and
                np.array_equal(iru, p["ir"]) and np.array_equal(ird, p["ir"])):
            continue  # the perturbation moved the selection: not differentiable there
        fd = (Lu - Ld) / (float(up[ix]) - float(dn[ix]))
        want = (dkp, dqp)[which][ix]
        assert fd == pytest.approx(want, rel=2e-3, abs=2e-4), (which, ix)
        checked += 1
    assert checked >= 20
