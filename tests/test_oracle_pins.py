"""Pins for the CPU oracle, against things other than the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed flat index, read-before-write, a wrong tie-break, a
missing softmax) fails at least one of them:

* a hand-worked two-token example (tests/golden/sdm_two_token_example.json);
* brute force over all N = S*S slot scores on tiny inputs with many ties, which
  pins the product-key identity topk(s1 (+) s2) = topk(topk(s1) (+) topk(s2));
* invariants of the update equations (alpha=1, beta=0 leaves M untouched;
  unselected rows never change; W=1, beta=1 writes v; R=1 reads one row);
* closed forms: one hot slot written every token (a scalar linear recurrence,
  compared with its product form) and W = R = N (every row follows its own
  scalar recurrence, weights from a softmax over all N slot scores).

Source of every equation: "Sparse Delta Memory (SDM)" technical summary,
gist.science/it/paper/2607.07386, section "Meccanismo Core", items 1-4.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sdm_two_token_example.json")


def _num(x, ln3):
    return ln3 if x == "ln3" else float(x)


def _load_example():
    with open(GOLDEN) as f:
        ex = json.load(f)
    ln3 = ex["ln3"]
    toks = ex["tokens"]
    kp = np.array([[[_num(x, ln3) for x in half] for half in t["kp"]] for t in toks], np.float32)
    qp = np.array([[[_num(x, ln3) for x in half] for half in t["qp"]] for t in toks], np.float32)
    v = np.array([t["v"] for t in toks], np.float32)
    alpha = np.array([t["alpha"] for t in toks], np.float32)
    beta = np.array([t["beta"] for t in toks], np.float32)
    return ex, kp, qp, v, alpha, beta


def test_two_token_worked_example():
    ex, kp, qp, v, alpha, beta = _load_example()
    M0 = np.array(ex["M0"], np.float64)
    res = oracle.forward(kp[None], qp[None], v[None], alpha[None], beta[None], M0[None],
                         ex["W"], ex["R"], n_threads=1)
    for t, tok in enumerate(ex["tokens"]):
        assert res["idx_w"][0, t].tolist() == tok["write_idx"]
        assert res["idx_r"][0, t].tolist() == tok["read_idx"]
        sw = res["sc_w"][0, t].astype(np.float64)
        ww = np.exp(sw - sw.max()) / np.exp(sw - sw.max()).sum()
        np.testing.assert_allclose(ww, tok["write_weights"], atol=1e-6)
        sr = res["sc_r"][0, t].astype(np.float64)
        rw = np.exp(sr - sr.max()) / np.exp(sr - sr.max()).sum()
        np.testing.assert_allclose(rw, tok["read_weights"], atol=1e-6)
        np.testing.assert_allclose(res["o"][0, t], tok["o"], atol=1e-6)
    np.testing.assert_allclose(res["M"][0], np.array(ex["M_final"]), atol=1e-6)
    # row 3 is never written: bit-identical to M0
    assert np.array_equal(res["M"][0, 3], M0[3])


def _tie_heavy(rng, shape):
    """Values from a small set of exactly representable numbers, with signed zeros,
    so that pair sums are exact in fp32 and ties are everywhere."""
    vals = np.array([-2.0, -1.0, -0.5, -0.0, 0.0, 0.5, 1.0, 1.5, 2.0], np.float32)
    return vals[rng.integers(0, len(vals), size=shape)]


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 7, 8, 16])
def test_select_matches_bruteforce_with_ties(S):
    rng = np.random.default_rng(100 + S)
    N = S * S
    for trial in range(40):
        K = int(rng.integers(1, N + 1))
        h = _tie_heavy(rng, (6, 2, S))
        i1, s1 = oracle.select(h, K, n_threads=1)
        i2, s2 = oracle.select_bruteforce(h, K)
        assert np.array_equal(i1, i2), (S, K, trial)
        assert np.array_equal(s1, s2), (S, K, trial)


def _bf16_round(x):
    """Round fp32 to the nearest bf16 (ties to even), returned as fp32."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("S,K", [(16, 1), (16, 8), (16, 16), (16, 40), (32, 8), (32, 32), (12, 144)])
def test_select_matches_bruteforce_bf16_gaussian(S, K):
    # bf16 sub-scores: every fp32 pair sum is exact, so the identity is exact.
    rng = np.random.default_rng(7 * S + K)
    h = _bf16_round(rng.standard_normal((50, 2, S)).astype(np.float32))
    i1, s1 = oracle.select(h, K, n_threads=2)
    i2, s2 = oracle.select_bruteforce(h, K)
    assert np.array_equal(i1, i2)
    assert np.array_equal(s1, s2)


def test_select_output_contract():
    rng = np.random.default_rng(3)
    S, K = 16, 24
    h = rng.standard_normal((20, 2, S)).astype(np.float32)
    idx, sc = oracle.select(h, K)
    for it in range(20):
        assert len(set(idx[it].tolist())) == K
        assert idx[it].min() >= 0 and idx[it].max() < S * S
        # scores are the fp32 sums of the two halves at (i, j) = divmod(flat, S)
        i, j = np.divmod(idx[it], S)
        assert np.array_equal(sc[it], (h[it, 0, i] + h[it, 1, j]).astype(np.float32))
        # ordered by (score desc, flat asc)
        for r in range(K - 1):
            assert sc[it, r] > sc[it, r + 1] or (sc[it, r] == sc[it, r + 1] and idx[it, r] < idx[it, r + 1])


def _random_case(rng, nh, T, S, dv, W, R):
    kp = rng.standard_normal((nh, T, 2, S)).astype(np.float32)
    qp = rng.standard_normal((nh, T, 2, S)).astype(np.float32)
    v = rng.standard_normal((nh, T, dv)).astype(np.float32)
    alpha = rng.uniform(0.9, 1.0, (nh, T)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (nh, T)).astype(np.float32)
    M0 = (0.02 * rng.standard_normal((nh, S * S, dv))).astype(np.float32)
    return kp, qp, v, alpha, beta, M0


def test_alpha_one_beta_zero_leaves_state_untouched():
    rng = np.random.default_rng(11)
    kp, qp, v, alpha, beta, M0 = _random_case(rng, 2, 30, 8, 4, 5, 3)
    alpha[:] = 1.0
    beta[:] = 0.0
    res = oracle.forward(kp, qp, v, alpha, beta, M0, 5, 3)
    assert np.array_equal(res["M"], M0.astype(np.float64))
    # the read is then a softmax-weighted sum of M0 rows
    for h in range(2):
        for t in range(30):
            s = res["sc_r"][h, t].astype(np.float64)
            w = np.exp(s - s.max())
            w /= w.sum()
            ref = (w[:, None] * M0[h, res["idx_r"][h, t]].astype(np.float64)).sum(0)
            np.testing.assert_allclose(res["o"][h, t], ref, rtol=1e-12, atol=1e-15)


def test_unselected_rows_unchanged():
    rng = np.random.default_rng(12)
    kp, qp, v, alpha, beta, M0 = _random_case(rng, 2, 40, 16, 8, 6, 4)
    res = oracle.forward(kp, qp, v, alpha, beta, M0, 6, 4)
    for h in range(2):
        written = np.zeros(256, bool)
        written[res["idx_w"][h].ravel()] = True
        assert (~written).sum() > 0
        assert np.array_equal(res["M"][h][~written], M0[h][~written].astype(np.float64))
        assert not np.array_equal(res["M"][h][written], M0[h][written].astype(np.float64))


def test_single_write_with_beta_one_stores_v():
    rng = np.random.default_rng(13)
    kp, qp, v, alpha, beta, M0 = _random_case(rng, 1, 25, 8, 6, 1, 1)
    beta[:] = 1.0
    idx_w, sc_w = oracle.select(kp, 1)
    idx_r, sc_r = oracle.select(qp, 1)
    M = M0.astype(np.float64)
    for t in range(25):
        # one token at a time so that the state after each token can be looked at
        oracle.scan(M, idx_w[:, t:t + 1], sc_w[:, t:t + 1], idx_r[:, t:t + 1], sc_r[:, t:t + 1],
                    v[:, t:t + 1], alpha[:, t:t + 1], beta[:, t:t + 1])
        np.testing.assert_allclose(M[0, idx_w[0, t, 0]], v[0, t], rtol=1e-15, atol=1e-15)
    # alpha = 0 as well: the slot is exactly v (the forget gate zeroes the old row)
    M = M0.astype(np.float64)
    alpha[:] = 0.0
    oracle.scan(M, idx_w, sc_w, idx_r, sc_r, v, alpha, beta)
    assert np.array_equal(M[0, idx_w[0, -1, 0]], v[0, -1].astype(np.float64))


def test_single_read_returns_the_row():
    rng = np.random.default_rng(14)
    kp, qp, v, alpha, beta, M0 = _random_case(rng, 1, 20, 8, 5, 4, 1)
    idx_w, sc_w = oracle.select(kp, 4)
    idx_r, sc_r = oracle.select(qp, 1)
    M = M0.astype(np.float64)
    for t in range(20):
        o = oracle.scan(M, idx_w[:, t:t + 1], sc_w[:, t:t + 1], idx_r[:, t:t + 1], sc_r[:, t:t + 1],
                        v[:, t:t + 1], alpha[:, t:t + 1], beta[:, t:t + 1])
        assert np.array_equal(o[0, 0], M[0, idx_r[0, t, 0]])


def test_closed_form_one_hot_slot():
    """W = R = 1 and a slot that wins every token: m_t = a_t m_{t-1} + b_t v_t with
    a_t = alpha_t (1 - beta_t), b_t = beta_t (k = 1).  Product form:
    m_T = (prod_t a_t) m_0 + sum_t b_t v_t prod_{s>t} a_s, and o_t = m_t."""
    rng = np.random.default_rng(15)
    T, S, dv = 60, 8, 3
    kp, qp, v, alpha, beta, M0 = _random_case(rng, 1, T, S, dv, 1, 1)
    kp[..., 0, 3] = 50.0
    kp[..., 1, 5] = 50.0
    qp[..., 0, 3] = 50.0
    qp[..., 1, 5] = 50.0
    hot = 3 * S + 5
    res = oracle.forward(kp, qp, v, alpha, beta, M0, 1, 1)
    assert (res["idx_w"] == hot).all() and (res["idx_r"] == hot).all()
    a = alpha[0].astype(np.float64) * (1.0 - beta[0].astype(np.float64))
    b = beta[0].astype(np.float64)
    m0 = M0[0, hot].astype(np.float64)
    for t in range(T):
        head = np.prod(a[: t + 1]) * m0
        tail = sum(b[s] * v[0, s].astype(np.float64) * np.prod(a[s + 1: t + 1]) for s in range(t + 1))
        np.testing.assert_allclose(res["o"][0, t], head + tail, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["M"][0, hot], head + tail, rtol=1e-11, atol=1e-13)
    others = np.arange(S * S) != hot
    assert np.array_equal(res["M"][0, others], M0[0, others].astype(np.float64))


def test_closed_form_every_row_selected():
    """W = R = N: every row i follows m_t[i] = alpha_t (1 - beta_t k_ti) m_{t-1}[i]
    + beta_t k_ti v_t, with k_t = softmax over all N outer-sum scores, and
    o_t = sum_i r_ti m_t[i] with r_t = softmax over all N read scores."""
    rng = np.random.default_rng(16)
    T, S, dv = 12, 3, 4
    N = S * S
    kp, qp, v, alpha, beta, M0 = _random_case(rng, 1, T, S, dv, N, N)
    kp[0, :, 1, :] *= 3.0  # make the two halves clearly different
    res = oracle.forward(kp, qp, v, alpha, beta, M0, N, N)
    m = M0[0].astype(np.float64).copy()
    for t in range(T):
        s_w = (kp[0, t, 0][:, None] + kp[0, t, 1][None, :]).astype(np.float32).ravel().astype(np.float64)
        k = np.exp(s_w - s_w.max())
        k /= k.sum()
        s_r = (qp[0, t, 0][:, None] + qp[0, t, 1][None, :]).astype(np.float32).ravel().astype(np.float64)
        r = np.exp(s_r - s_r.max())
        r /= r.sum()
        at, bt = float(alpha[0, t]), float(beta[0, t])
        m = (at * (1.0 - bt * k))[:, None] * m + (bt * k)[:, None] * v[0, t].astype(np.float64)[None, :]
        np.testing.assert_allclose(res["o"][0, t], (r[:, None] * m).sum(0), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["M"][0], m, rtol=1e-11, atol=1e-13)


def test_scan_rejects_out_of_range_index():
    M = np.zeros((1, 4, 2))
    iw = np.array([[[0, 4]]], np.int32)
    with pytest.raises(ValueError):
        oracle.scan(M, iw, np.zeros((1, 1, 2), np.float32), np.zeros((1, 1, 1), np.int32),
                    np.zeros((1, 1, 1), np.float32), np.zeros((1, 1, 2), np.float32),
                    np.ones((1, 1), np.float32), np.ones((1, 1), np.float32))
