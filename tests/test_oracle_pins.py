"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test here checks the oracle against something other than itself: a
value printed on the pages, a hand-worked case, a closed form, a textbook
or library routine (scipy softmax, numpy searchsorted, torch's
scaled_dot_product_attention), an invariant, or a statistical property
(losslessness, the mean acceptance length).  A plausible slip in the oracle
(a dropped term, a swapped P/Q, a wrong row, u <= alpha instead of u < alpha,
an ignored temperature or scale, a wrong GQA head map, a mask that leaks
across branches) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- N_async
def test_n_async_printed_value():
    g = json.load(open(os.path.join(GOLD, "n_async.json")))
    assert oracle.n_async(g["B"], g["C"], g["F"]) == g["N_async"] == 384


@pytest.mark.parametrize("C", [1, 2, 3, 4, 8, 12, 16])
@pytest.mark.parametrize("F", [1, 2, 3, 5])
def test_async_layout_fills_budget(C, F):
    # the generator's branch layout has exactly the pages' budget of tokens,
    # and one head per segment
    segs = W.async_segments(16, C, F)
    assert int(segs[:, 1].sum()) == oracle.n_async(16, C, F)
    assert len(segs) == (C - 1) * F + 2
    assert oracle.check_segments(segs, [0, int(segs[:, 1].sum())], [0, len(segs)]) == 0


# ---------------------------------------------------------------- tau
def test_tau_closed_forms():
    B = 16
    assert oracle.expected_tau(np.ones(B - 1)) == pytest.approx(B)
    a = np.full(B - 1, 0.7)
    a[0] = 0.0
    assert oracle.expected_tau(a) == pytest.approx(1.0)
    for c in (0.1, 0.5, 0.9):
        closed = 1 + c * (1 - c ** (B - 1)) / (1 - c)
        assert oracle.expected_tau(np.full(B - 1, c)) == pytest.approx(closed, rel=1e-12)
    # hand-worked: V=2, P=(1/2,1/2), Q=(1,0) at every position => a_j = 1/2; B=4
    assert oracle.expected_tau([0.5, 0.5, 0.5]) == pytest.approx(1.875)


def test_accept_probs_special_cases_and_tau():
    # P = Q: every draft is accepted (a = 1, tau = B); disjoint supports: a = 0
    # (tau = 1); the hand case of test_tau_closed_forms: V = 2, P = (1/2, 1/2),
    # Q = (1, 0) gives a = 1/2 and tau = 1.875 at B = 4
    B, V = 4, 2
    eq = np.array([[[0.3, -1.2]] * B], np.float32)
    r = oracle.accept_probs(dict(target=eq, draft=eq[:, : B - 1], dtype=W.DT_F32, R=1, B=B, V=V))
    np.testing.assert_allclose(r["accept_prob"], 1.0, rtol=1e-12)
    assert r["tau"][0] == pytest.approx(B)
    big = 1e4
    disj_t = np.array([[[big, -big]] * B], np.float32)
    disj_d = np.array([[[-big, big]] * (B - 1)], np.float32)
    r = oracle.accept_probs(dict(target=disj_t, draft=disj_d, dtype=W.DT_F32, R=1, B=B, V=V))
    assert r["accept_prob"].max() < 1e-300 and r["tau"][0] == pytest.approx(1.0)
    half = np.array([[[0.0, 0.0]] * B], np.float32)
    one = np.array([[[big, -big]] * (B - 1)], np.float32)
    r = oracle.accept_probs(dict(target=half, draft=one, dtype=W.DT_F32, R=1, B=B, V=V))
    np.testing.assert_allclose(r["accept_prob"], 0.5, rtol=1e-12)
    assert r["tau"][0] == pytest.approx(1.875)
    np.testing.assert_allclose(r["survival"][0], [0.5, 0.25, 0.125], rtol=1e-12)


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_accept_probs_match_library_softmax(T):
    x, z = _rows(200, 8, seed=35)
    P = scipy.special.softmax(x.astype(np.float64) / T, axis=-1)
    Q = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    a = np.minimum(P[: 7], Q).sum(-1)
    r = oracle.accept_probs(dict(target=x[None], draft=z[None], dtype=W.DT_F32, R=1, B=8, V=200, temperature=T))
    np.testing.assert_allclose(r["accept_prob"][0], a, rtol=1e-12)
    assert r["tau"][0] == pytest.approx(oracle.expected_tau(a), rel=1e-12)


# ---------------------------------------------------------------- hand-worked verify cases
def _case_inputs(c):
    B, V = c["B"], c["V"]
    return dict(target=np.array(c["target"], np.float32).reshape(1, B, V),
                draft=np.array(c["draft"], np.float32).reshape(1, B - 1, V), dtype=W.DT_F32,
                y=np.array(c["y"], np.int32).reshape(1, B - 1),
                u_accept=np.array(c["u_accept"], np.float32).reshape(1, B - 1),
                u_sample=np.array([c["u_sample"]], np.float32), R=1, B=B, V=V,
                temperature=c["T"])


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "verify_hand.json")))["cases"],
                         ids=lambda c: c["name"])
def test_verify_hand_worked(case):
    r = oracle.spec_verify(_case_inputs(case))
    np.testing.assert_allclose(r["alpha"][0], case["alpha"], rtol=1e-6, atol=1e-7)
    assert int(r["accept_len"][0]) == case["accept_len"]
    n = case["accept_len"] + 1
    assert int(r["num_tokens"][0]) == n
    assert r["out_tokens"][0, :n].tolist() == case["tokens"]
    assert (r["out_tokens"][0, n:] == -1).all()
    # the near-tie margins and the zero-residual fallback, worked out by hand
    # (abs 1e-7: the uniforms are float32, within 6e-8 of the decimals written)
    assert r["margin_accept"][0] == pytest.approx(case["margin_accept"], abs=1e-7)
    assert r["margin_sample"][0] == pytest.approx(case["margin_sample"], abs=1e-7)
    assert int(r["used_fallback"][0]) == case["used_fallback"]


def _margins_by_library(inp):
    """The oracle's margins restated with library routines: scipy softmax for
    P, Q and alpha, numpy cumsum/searchsorted for the inverse CDF."""
    R, B, V, T = inp["R"], inp["B"], inp["V"], inp["temperature"]
    P = scipy.special.softmax(inp["target"].astype(np.float64) / T, axis=-1)
    Q = scipy.special.softmax(inp["draft"].astype(np.float64) / T, axis=-1)
    ma, ms, fb, tok = np.zeros(R), np.zeros(R), np.zeros(R, np.int32), np.zeros(R, np.int32)
    for r in range(R):
        y = inp["y"][r]
        p, q = P[r, np.arange(B - 1), y], Q[r, np.arange(B - 1), y]
        al = np.minimum(1.0, p / q)
        u = inp["u_accept"][r].astype(np.float64)
        rej = np.nonzero(~(u < al))[0]
        a = int(rej[0]) if len(rej) else B - 1
        decided = np.arange(min(a + 1, B - 1))
        ma[r] = np.abs(u[decided] - al[decided]).min()
        w = np.maximum(P[r, a] - Q[r, a], 0.0) if a < B - 1 else P[r, B - 1]
        if not w.sum() > 0:
            fb[r], w = 1, P[r, a]
        c = np.cumsum(w)
        S = c[-1]
        x = float(inp["u_sample"][r]) * S
        v = min(int(np.searchsorted(c, x, side="right")), V - 1)
        lo = x - (c[v - 1] if v > 0 else 0.0)
        ms[r] = min(lo, c[v] - x) / S
        tok[r] = v
    return ma, ms, fb, tok


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_margins_match_library_restatement(T):
    # random rows whose acceptance uniforms sit close to alpha and whose sample
    # uniforms sit close to a CDF step: the oracle's two margins and tokens
    # equal the scipy/numpy restatement
    rng = np.random.default_rng(61)
    R, B, V = 400, 5, 40
    x = (rng.standard_normal((R, B, V)) * 2).astype(np.float32)
    z = (x[:, : B - 1] + rng.standard_normal((R, B - 1, V)) * 0.8).astype(np.float32)
    Q = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    y = np.array([[rng.choice(V, p=Q[r, j]) for j in range(B - 1)] for r in range(R)], np.int32)
    inp = dict(target=x, draft=z, dtype=W.DT_F32, y=y, R=R, B=B, V=V, temperature=T,
               u_accept=rng.random((R, B - 1)).astype(np.float32),
               u_sample=rng.random(R).astype(np.float32))
    P = scipy.special.softmax(x.astype(np.float64) / T, axis=-1)
    al = np.minimum(1.0, P[np.arange(R)[:, None], np.arange(B - 1)[None], y] /
                    Q[np.arange(R)[:, None], np.arange(B - 1)[None], y])
    near = rng.random((R, B - 1)) < 0.3  # some uniforms a known small distance from alpha
    inp["u_accept"] = np.where(near, np.clip(al + rng.choice([-1, 1], (R, B - 1)) * 1e-4, 0, 0.999999),
                               inp["u_accept"]).astype(np.float32)
    r = oracle.spec_verify(inp)
    ma, ms, fb, tok = _margins_by_library(inp)
    np.testing.assert_allclose(r["margin_accept"], ma, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["margin_sample"], ms, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(r["used_fallback"], fb)
    keep = ms > 1e-9
    np.testing.assert_array_equal(r["out_tokens"][np.arange(R), r["accept_len"]][keep], tok[keep])
    assert (r["margin_accept"] < 2e-4).sum() > 50 and (r["margin_sample"] < 0.05).sum() > 20


def test_zero_residual_falls_back_to_P_in_distribution():
    # identical target and draft rows with u = 1 (outside [0, 1)) reject with a
    # residual of exactly zero: the token then follows P at that row
    V, B, R = 12, 3, 100_000
    x, _ = _rows(V, B, seed=71)
    inp = _fixed_rows_inputs(x, x[: B - 1].copy(), 1.0, R, seed=72)
    inp["u_accept"][:, 1] = 1.0
    r = oracle.spec_verify(inp)
    assert (r["accept_len"] == 1).all() and (r["used_fallback"] == 1).all()
    P = scipy.special.softmax(x.astype(np.float64), axis=-1)
    assert _chi2_p(r["out_tokens"][:, 1], P[1]) > 1e-4


# ---------------------------------------------------------------- AWL weights
@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "awl_hand.json")))["cases"],
                         ids=lambda c: c["name"])
def test_awl_weights_hand_worked(case):
    r = oracle.spec_verify(dict(_case_inputs(dict(case, u_accept=[0.5] * (case["B"] - 1), u_sample=0.5))))
    # (rtol 1e-6: the logits are float32 roundings of the logarithms written)
    np.testing.assert_allclose(r["alpha"][0], case["alpha"], rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(oracle.awl_weights(r["alpha"])[0], case["awl"], rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_awl_weight_is_the_probability_of_reaching_a_position(T):
    # fixed rows and fixed drafted tokens, fresh acceptance uniforms each
    # trial: the fraction of trials whose accepted length is at least k (the
    # verification reached position k) estimates w_k
    V, B, R = 24, 6, 200_000
    x, z = _rows(V, B, seed=81, sigma=0.7)
    Q = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    rng = np.random.default_rng(82)
    y = np.array([rng.choice(V, p=Q[j]) for j in range(B - 1)], np.int32)
    inp = _fixed_rows_inputs(x, z, T, R, seed=83)
    inp["y"] = np.ascontiguousarray(np.broadcast_to(y, (R, B - 1)))
    r = oracle.spec_verify(inp)
    w = oracle.awl_weights(r["alpha"][:1])[0]
    for k in range(B - 1):
        emp = (r["accept_len"] >= k).mean()
        se = max(np.sqrt(w[k] * (1 - w[k]) / R), 1e-9)
        assert abs(emp - w[k]) <= 5 * se + 1e-12, (k, emp, w[k])
    assert 0.05 < w[-1] < 0.95  # the case exercises partial acceptance


# ---------------------------------------------------------------- greedy (temperature 0)
@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "verify_greedy.json")))["cases"],
                         ids=lambda c: c["name"])
def test_greedy_hand_worked(case):
    B, V = case["B"], case["V"]
    r = oracle.greedy_verify(dict(target=np.array(case["target"], np.float32).reshape(1, B, V), dtype=W.DT_F32,
                                  y=np.array(case["y"], np.int32).reshape(1, B - 1), R=1, B=B, V=V))
    assert r["argmax"][0].tolist() == case["argmax"]
    assert r["accept"][0].tolist() == case["accept"]
    assert int(r["accept_len"][0]) == case["accept_len"]
    n = case["accept_len"] + 1
    assert int(r["num_tokens"][0]) == n
    assert r["out_tokens"][0, :n].tolist() == case["tokens"]
    assert (r["out_tokens"][0, n:] == -1).all()


def test_greedy_is_the_zero_temperature_limit_of_sampling():
    # distinct logits 0.1 apart: at T = 1e-3 the softmaxes are point masses to
    # within exp(-100), so the sampling rule with any uniforms in (0, 1)
    # accepts exactly the drafts that are the target's argmax and emits the
    # target's argmax; the draft tokens are the draft rows' argmax
    rng = np.random.default_rng(31)
    R, B, V = 64, 6, 40
    tgt = np.stack([[rng.permutation(V) * 0.1 for _ in range(B)] for _ in range(R)]).astype(np.float32)
    dr = tgt[:, : B - 1].copy()
    redo = rng.random((R, B - 1)) < 0.35  # some draft rows disagree with the target
    dr[redo] = np.stack([rng.permutation(V) * 0.1 for _ in range(int(redo.sum()))]).astype(np.float32)
    y = dr.argmax(-1).astype(np.int32)
    u = (rng.integers(1, 1 << 24, size=(R, B)) * 2.0 ** -24).astype(np.float32)  # never 0
    samp = oracle.spec_verify(dict(target=tgt, draft=dr, dtype=W.DT_F32, y=y, u_accept=u[:, : B - 1].copy(),
                                   u_sample=u[:, B - 1].copy(), R=R, B=B, V=V, temperature=1e-3))
    gr = oracle.greedy_verify(dict(target=tgt, dtype=W.DT_F32, y=y, R=R, B=B, V=V))
    np.testing.assert_array_equal(gr["accept_len"], samp["accept_len"])
    np.testing.assert_array_equal(gr["out_tokens"], samp["out_tokens"])
    assert (gr["accept_len"] < B - 1).any() and (gr["accept_len"] == B - 1).any()  # both outcomes occur


@pytest.mark.parametrize("dt", [W.DT_F32, W.DT_BF16])
def test_greedy_matches_first_max_scan_with_many_ties(dt):
    # integer logits in 0..3 make ties common: numpy's argmax returns the
    # first maximum, the reading the oracle follows
    rng = np.random.default_rng(32)
    R, B, V = 50, 5, 23
    vals = rng.integers(0, 4, size=(R, B, V)).astype(np.float32)
    g = vals.argmax(-1)
    y = np.where(rng.random((R, B - 1)) < 0.7, g[:, : B - 1], rng.integers(0, V, size=(R, B - 1))).astype(np.int32)
    tgt = W.bf16_bits(vals) if dt == W.DT_BF16 else vals
    r = oracle.greedy_verify(dict(target=tgt, dtype=dt, y=y, R=R, B=B, V=V))
    np.testing.assert_array_equal(r["argmax"], g)
    for i in range(R):
        a = 0
        while a < B - 1 and y[i, a] == g[i, a]:
            a += 1
        assert r["accept_len"][i] == a
        assert r["out_tokens"][i].tolist() == y[i, :a].tolist() + [g[i, a]] + [-1] * (B - 1 - a)
    np.testing.assert_array_equal(r["accept"], (y == g[:, : B - 1]).astype(np.float64))


# ---------------------------------------------------------------- branch construction
@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "build_branches.json")))["cases"],
                         ids=lambda c: c["name"])
def test_build_branches_hand_worked(case):
    B, V, C, F = case["B"], case["V"], case["C"], case["F"]
    bg = None if case["bonus_guess"] is None else np.array([case["bonus_guess"]], np.int32)
    r = oracle.build_branches(dict(draft=np.array(case["draft"], np.float32).reshape(1, B - 1, V), dtype=W.DT_F32,
                                   y=np.array(case["y"], np.int32).reshape(1, B - 1), bonus_guess=bg,
                                   R=1, B=B, V=V, C=C, F=F))
    assert r["anchors"][0].tolist() == case["anchors"]
    assert r["heads"][0].tolist() == case["heads"]
    assert r["head_len"][0].tolist() == case["head_len"]


@pytest.mark.parametrize("B,C,F", [(16, 12, 2), (16, 4, 1), (16, 16, 5), (8, 3, 2), (4, 1, 3)])
def test_build_branches_segments_are_the_async_layout(B, C, F):
    # the segment rows equal the layout whose size is the printed N_async
    R, V = 3, 50
    rng = np.random.default_rng(33)
    r = oracle.build_branches(dict(draft=rng.standard_normal((R, B - 1, V)).astype(np.float32), dtype=W.DT_F32,
                                   y=rng.integers(0, V, size=(R, B - 1)).astype(np.int32), R=R, B=B, V=V, C=C, F=F))
    lay = W.async_segments(B, C, F)
    M = len(lay)
    assert M == (C - 1) * F + 2 and int(lay[:, 1].sum()) == oracle.n_async(B, C, F)
    np.testing.assert_array_equal(r["segs"], np.concatenate([lay] * R))
    np.testing.assert_array_equal(r["cu_q"], np.arange(R + 1) * M * B)
    np.testing.assert_array_equal(r["cu_seg"], np.arange(R + 1) * M)


@pytest.mark.parametrize("dt", [W.DT_F32, W.DT_BF16])
def test_build_branches_anchors_match_a_sort(dt):
    # integer logits make ties common; a stable sort by (-logit, index) with
    # y removed gives the anchors; every head is y's prefix then the anchor
    rng = np.random.default_rng(34)
    R, B, V, C, F = 20, 8, 30, 6, 3
    vals = rng.integers(0, 5, size=(R, B - 1, V)).astype(np.float32)
    y = rng.integers(0, V, size=(R, B - 1)).astype(np.int32)
    dr = W.bf16_bits(vals) if dt == W.DT_BF16 else vals
    bg = rng.integers(0, V, size=R).astype(np.int32)
    r = oracle.build_branches(dict(draft=dr, dtype=dt, y=y, bonus_guess=bg, R=R, B=B, V=V, C=C, F=F))
    for i in range(R):
        for p in range(C - 1):
            order = [v for v in np.lexsort((np.arange(V), -vals[i, p])) if v != y[i, p]]
            assert r["anchors"][i, p].tolist() == order[:F]
            for f in range(F):
                k = 1 + p * F + f
                assert r["head_len"][i, k] == p + 1
                assert r["heads"][i, k, :p].tolist() == y[i, :p].tolist()
                assert r["heads"][i, k, p] == order[f] and (r["heads"][i, k, p + 1:] == -1).all()
        assert r["head_len"][i, -1] == B and r["heads"][i, -1].tolist() == y[i].tolist() + [bg[i]]


# ---------------------------------------------------------------- statistics helpers
def _fixed_rows_inputs(x, z, T, R, seed):
    """R trials of one fixed verification problem: target rows x [B, V], draft
    rows z [B-1, V]; each trial draws its own draft tokens y_j ~ Q_j (scipy
    softmax) and its own uniforms."""
    B, V = x.shape
    rng = np.random.default_rng(seed)
    Qd = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    y = np.stack([rng.choice(V, size=R, p=Qd[j]) for j in range(B - 1)], axis=1).astype(np.int32)
    u = W.uniform24(rng, (R, B))
    return dict(target=np.broadcast_to(x, (R, B, V)).copy(), draft=np.broadcast_to(z, (R, B - 1, V)).copy(),
                dtype=W.DT_F32, y=y, u_accept=np.ascontiguousarray(u[:, :B - 1]),
                u_sample=np.ascontiguousarray(u[:, B - 1]), R=R, B=B, V=V, temperature=T)


def _chi2_p(tokens, probs):
    V = len(probs)
    obs = np.bincount(tokens, minlength=V).astype(np.float64)
    exp = probs * obs.sum()
    keep = exp > 0
    assert obs[~keep].sum() == 0, "token with zero target probability was emitted"
    return scipy.stats.chisquare(obs[keep], exp[keep]).pvalue


def _rows(V, B, seed, sigma=1.0, scale=1.5):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((B, V)) * scale).astype(np.float32)
    z = (x[: B - 1] + rng.standard_normal((B - 1, V)) * sigma).astype(np.float32)
    return x, z


# ---------------------------------------------------------------- mean acceptance length (MC)
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_tau_monte_carlo_matches_closed_form(T):
    # a_j = sum_v min(P_j(v), Q_j(v)) is the per-position acceptance
    # probability of speculative sampling (1 - total variation distance);
    # the pages' MAT formula then gives E[a + 1].
    V, B, R = 8, 5, 200_000
    x, z = _rows(V, B, seed=11, sigma=1.2)
    inp = _fixed_rows_inputs(x, z, T, R, seed=5)
    r = oracle.spec_verify(inp)
    P = scipy.special.softmax(x.astype(np.float64) / T, axis=-1)
    Q = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    a = np.minimum(P[: B - 1], Q).sum(axis=-1)
    tau = 1.0 + sum(np.prod(a[: k + 1]) for k in range(B - 1))
    n = r["num_tokens"].astype(np.float64)
    se = n.std() / np.sqrt(R)
    assert abs(n.mean() - tau) < 5 * se, (n.mean(), tau, se)
    # per-position survival as well (catches an index slip that keeps the mean)
    for k in range(1, B):
        s_emp = (r["accept_len"] >= k).mean()
        s_true = np.prod(a[:k])
        assert abs(s_emp - s_true) < 5 * np.sqrt(s_true * (1 - s_true) / R) + 1e-12


# ---------------------------------------------------------------- losslessness (chi-square)
@pytest.mark.slow
@pytest.mark.parametrize("T", [1.0, 2.0])
def test_lossless_chi_square(T):
    # D3D/DScout "Background": the output distribution equals the target's.
    # First emitted token ~ P_1; second emitted token given the first draft
    # was accepted ~ P_2.  V <= 64, >= 10^6 trials, flag at p < 1e-4.
    V, B = 16, 3
    x, z = _rows(V, B, seed=3, sigma=1.0)
    P = scipy.special.softmax(x.astype(np.float64) / T, axis=-1)
    first, second = [], []
    for chunk in range(5):
        inp = _fixed_rows_inputs(x, z, T, 200_000, seed=100 + chunk)
        r = oracle.spec_verify(inp)
        first.append(r["out_tokens"][:, 0])
        ok = r["accept_len"] >= 1
        second.append(r["out_tokens"][ok, 1])
    first, second = np.concatenate(first), np.concatenate(second)
    assert len(first) == 1_000_000
    assert _chi2_p(first, P[0]) > 1e-4
    assert _chi2_p(second, P[1]) > 1e-4


def test_lossless_detects_a_wrong_rule():
    # the chi-square check has power: plain "accept if y == argmax" style
    # outputs (here: always emitting the draft token) are not ~ P_1
    V, B = 16, 2
    x, z = _rows(V, B, seed=3, sigma=1.0)
    P = scipy.special.softmax(x.astype(np.float64), axis=-1)
    inp = _fixed_rows_inputs(x, z, 1.0, 200_000, seed=9)
    assert _chi2_p(inp["y"][:, 0], P[0]) < 1e-4


# ---------------------------------------------------------------- special cases
def test_equal_distributions_always_accept_and_bonus_is_P_B():
    V, B, R = 12, 4, 200_000
    x, _ = _rows(V, B, seed=21)
    inp = _fixed_rows_inputs(x, x[: B - 1].copy(), 1.0, R, seed=22)
    r = oracle.spec_verify(inp)
    assert (r["accept_len"] == B - 1).all()
    assert (r["alpha"] == 1.0).all()
    P = scipy.special.softmax(x.astype(np.float64), axis=-1)
    assert _chi2_p(r["out_tokens"][:, B - 1], P[B - 1]) > 1e-4
    np.testing.assert_array_equal(r["out_tokens"][:, : B - 1], inp["y"])


def test_disjoint_support_always_rejects_first_and_samples_P1():
    V, B, R = 16, 3, 200_000
    rng = np.random.default_rng(31)
    x = rng.standard_normal((B, V)).astype(np.float32)
    z = rng.standard_normal((B - 1, V)).astype(np.float32)
    x[0, 8:] = -10000.0   # P_1 lives on tokens 0..7
    z[0, :8] = -10000.0   # Q_1 lives on tokens 8..15
    inp = _fixed_rows_inputs(x, z, 1.0, R, seed=32)
    r = oracle.spec_verify(inp)
    assert (r["accept_len"] == 0).all()
    assert (r["alpha"][:, 0] == 0.0).all()
    P = scipy.special.softmax(x.astype(np.float64), axis=-1)
    assert _chi2_p(r["out_tokens"][:, 0], P[0]) > 1e-4


def test_one_token_vocabulary():
    """V = 1: every distribution is the point mass on token 0 whatever the
    logits and the temperature, so alpha = 1 > u for every u in [0, 1): all
    drafts are accepted and the bonus is token 0; the greedy argmax is 0;
    a_j = 1, S(k) = 1 and tau = B.  No anchor exists besides the drafted
    token, so F > 0 is rejected; with F = 0 the pass holds only the block
    under verification and the all-accept block."""
    R, B, V, T = 3, 5, 1, 0.7
    rng = np.random.default_rng(3)
    tgt = (rng.standard_normal((R, B, V)) * 5).astype(np.float32)
    dr = (rng.standard_normal((R, B - 1, V)) * 5).astype(np.float32)
    y = np.zeros((R, B - 1), np.int32)
    inp = dict(target=tgt, draft=dr, dtype=W.DT_F32, y=y, R=R, B=B, V=V, temperature=T,
               u_accept=np.full((R, B - 1), np.nextafter(np.float32(1), np.float32(0))),
               u_sample=rng.random(R).astype(np.float32))
    r = oracle.spec_verify(inp)
    assert (r["alpha"] == 1.0).all() and (r["p"] == 1.0).all() and (r["q"] == 1.0).all()
    assert (r["accept_len"] == B - 1).all() and (r["num_tokens"] == B).all()
    assert (r["out_tokens"] == 0).all() and not r["used_fallback"].any()
    g = oracle.greedy_verify(inp)
    assert (g["argmax"] == 0).all() and (g["accept"] == 1.0).all()
    assert (g["accept_len"] == B - 1).all() and (g["out_tokens"] == 0).all()
    a = oracle.accept_probs(inp)
    assert (a["accept_prob"] == 1.0).all() and (a["survival"] == 1.0).all() and (a["tau"] == B).all()
    br = dict(draft=dr, dtype=W.DT_F32, y=y, R=R, B=B, V=V, C=3, bonus_guess=np.zeros(R, np.int32))
    with pytest.raises(ValueError):
        oracle.build_branches(dict(br, F=1))
    b = oracle.build_branches(dict(br, F=0))
    assert b["head_len"].tolist() == [[0, B]] * R
    assert (b["heads"][:, 1] == 0).all() and (b["heads"][:, 0] == -1).all()
    assert b["segs"].tolist() == [[0, B, W.SEG_CAUSAL, -1, 0], [B, B, W.SEG_BIDIR, 0, B]] * R
    assert b["cu_q"].tolist() == [2 * B * r for r in range(R + 1)]


def test_rejection_never_emits_rejected_token():
    V, B, R = 10, 6, 50_000
    x, z = _rows(V, B, seed=41, sigma=2.0)
    inp = _fixed_rows_inputs(x, z, 1.0, R, seed=42)
    r = oracle.spec_verify(inp)
    rej = np.nonzero(r["accept_len"] < B - 1)[0]
    assert len(rej) > 1000
    a = r["accept_len"][rej]
    assert (r["out_tokens"][rej, a] != inp["y"][rej, a]).all()
    assert not r["used_fallback"].any()


def test_inverse_cdf_matches_searchsorted():
    # Bonus path (P = Q in rows 1..B-1) and residual path with disjoint
    # support (residual = P_1): the emitted token equals numpy's
    # searchsorted over the cumulative target probabilities (scipy softmax).
    rng = np.random.default_rng(51)
    for trial in range(200):
        V = int(rng.integers(2, 300))
        B = int(rng.integers(2, 6))
        x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
        if trial % 2 == 0:
            z = x[: B - 1].copy()
            row = B - 1
        else:
            z = rng.standard_normal((B - 1, V)).astype(np.float32)
            cut = int(rng.integers(1, V)) if V > 1 else 1
            x[0, cut:] = -10000.0
            z[0, :cut] = -10000.0
            row = 0
        inp = _fixed_rows_inputs(x, z, 1.0, 64, seed=trial)
        r = oracle.spec_verify(inp)
        P = scipy.special.softmax(x[row].astype(np.float64))
        c = np.cumsum(P)
        ref = np.searchsorted(c, inp["u_sample"].astype(np.float64) * c[-1], side="right")
        ref = np.minimum(ref, V - 1)
        pos = r["accept_len"]
        got = r["out_tokens"][np.arange(64), pos]
        keep = r["margin_sample"] > 1e-9
        assert keep.sum() > 50
        np.testing.assert_array_equal(got[keep], ref[keep])


def test_alpha_p_q_match_library_softmax():
    inp = W.verify_inputs(**W.CONFIGS["tiny"], seed=3)
    r = oracle.spec_verify(inp)
    P = scipy.special.softmax(inp["target"].astype(np.float64), axis=-1)
    Q = scipy.special.softmax(inp["draft"].astype(np.float64), axis=-1)
    idx = np.arange(inp["B"] - 1)
    p = P[0, idx, inp["y"][0]]
    q = Q[0, idx, inp["y"][0]]
    np.testing.assert_allclose(r["p"][0], p, rtol=1e-12)
    np.testing.assert_allclose(r["q"][0], q, rtol=1e-12)
    np.testing.assert_allclose(r["alpha"][0], np.minimum(1.0, p / q), rtol=1e-12)


def test_bf16_logits_decode_exactly():
    inp = W.verify_inputs(R=2, B=4, V=64, logits=W.DT_BF16, seed=4)
    r16 = oracle.spec_verify(inp)
    f32 = dict(inp, target=W.bf16_to_f32(inp["target"]), draft=W.bf16_to_f32(inp["draft"]), dtype=W.DT_F32)
    r32 = oracle.spec_verify(f32)
    for k in ("accept_len", "out_tokens", "alpha"):
        np.testing.assert_array_equal(r16[k], r32[k])


# ---------------------------------------------------------------- attention
def _f64(bits):
    return torch.from_numpy(W.bf16_to_f32(bits).astype(np.float64))


def _sdpa(q, k, v, scale, causal=False):
    """torch SDPA in fp64; q [n, H, d], k/v [m, Hkv, d] with GQA expansion."""
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    qt, kt, vt = (t.permute(1, 0, 2) for t in (q, k, v))
    mask = None
    if causal:
        n, m = q.shape[0], k.shape[0]
        mask = torch.ones(n, m, dtype=torch.bool).tril(diagonal=m - n)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("B,C,F,L,Hq,Hkv,d,scale", [
    (4, 3, 2, 8, 4, 2, 8, None), (4, 4, 1, 5, 2, 2, 16, 0.3), (3, 2, 3, 1, 8, 2, 4, None),
    (6, 4, 2, 0, 4, 1, 8, None)])
def test_packing_invariance_vs_sdpa(B, C, F, L, Hq, Hkv, d, scale):
    """Each branch's rows equal an independent attention of that block over
    [prefix | c_0 .. c_r | own block]; the current segment equals causal
    attention over [prefix | current block] (torch SDPA, fp64, GQA by
    repeat_interleave)."""
    inp = W.attn_inputs(R=1, L=L, Hq=Hq, Hkv=Hkv, d=d, B=B, C=C, F=F, layout="async", seed=7)
    if scale is not None:
        inp["scale"] = scale
    out = oracle.packed_attn(inp)
    q, kp, vp, kn, vn = (_f64(inp[k]) for k in ("q", "kp", "vp", "kn", "vn"))
    s = inp["scale"]
    for g in inp["segs"]:
        q0, n, mode, par, plen = (int(t) for t in g)
        rows = slice(q0, q0 + n)
        if par >= 0:
            p0 = int(inp["segs"][par][0])
            ks = torch.cat([kp, kn[p0:p0 + plen], kn[rows]])
            vs = torch.cat([vp, vn[p0:p0 + plen], vn[rows]])
        else:
            ks, vs = torch.cat([kp, kn[rows]]), torch.cat([vp, vn[rows]])
        ref = _sdpa(q[rows], ks, vs, s, causal=(mode == W.SEG_CAUSAL))
        np.testing.assert_allclose(out[rows], ref, rtol=1e-10, atol=1e-12)


def test_single_block_is_noncausal_and_single_causal_is_textbook():
    inp = W.attn_inputs(R=1, L=12, Hq=4, Hkv=2, d=8, B=8, layout="block", seed=8)
    out = oracle.packed_attn(inp)
    q, kp, vp, kn, vn = (_f64(inp[k]) for k in ("q", "kp", "vp", "kn", "vn"))
    ref = _sdpa(q, torch.cat([kp, kn]), torch.cat([vp, vn]), inp["scale"])
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    inp2 = W.attn_inputs(R=1, L=12, Hq=4, Hkv=2, d=8, B=8, seed=8,
                         segs=np.array([[0, 8, W.SEG_CAUSAL, -1, 0]]))
    out2 = oracle.packed_attn(inp2)
    ref2 = _sdpa(q, torch.cat([kp, kn]), torch.cat([vp, vn]), inp2["scale"], causal=True)
    np.testing.assert_allclose(out2, ref2, rtol=1e-10, atol=1e-12)


def _random_segments(rng, n_seg):
    rows, q = [], 0
    causal = []
    for s in range(n_seg):
        ln = int(rng.integers(1, 6))
        mode = int(rng.integers(0, 2))
        par, plen = -1, 0
        if causal and rng.random() < 0.7:
            par = int(rng.choice(causal))
            plen = int(rng.integers(0, rows[par][1] + 1))
        rows.append([q, ln, mode, par, plen])
        if mode == W.SEG_CAUSAL and par == -1:
            causal.append(s)
        q += ln
    return np.array(rows, np.int32)


def test_predicate_equals_dense_mask_random_tables():
    rng = np.random.default_rng(61)
    for t in range(40):
        segs = _random_segments(rng, int(rng.integers(1, 9)))
        N = int(segs[-1, 0] + segs[-1, 1])
        L = int(rng.integers(0, 9))
        inp = W.attn_inputs(R=1, L=L, Hq=2, Hkv=1, d=4, seed=t, segs=segs)
        np.testing.assert_allclose(oracle.packed_attn(inp), oracle.dense_attn(inp), rtol=1e-12, atol=1e-14)
        m = oracle.dense_mask(segs, L, N)
        assert m[:, :L].all()
        # no cross-branch leak: a row never sees a later segment's tokens
        for g in segs:
            q0, n = int(g[0]), int(g[1])
            assert not m[q0:q0 + n, L + q0 + n:].any()


def test_ragged_batch_equals_requests_alone():
    segs = W.async_segments(4, 3, 2)
    inp = W.attn_inputs(R=3, L=(0, 9), Hq=4, Hkv=2, d=8, seed=9, segs=segs)
    out = oracle.packed_attn(inp)
    for r in range(3):
        p0, p1 = inp["cu_prefix"][r], inp["cu_prefix"][r + 1]
        q0, q1 = inp["cu_q"][r], inp["cu_q"][r + 1]
        one = dict(inp, R=1, q=inp["q"][q0:q1], kp=inp["kp"][p0:p1], vp=inp["vp"][p0:p1],
                   kn=inp["kn"][q0:q1], vn=inp["vn"][q0:q1], segs=segs,
                   cu_prefix=np.array([0, p1 - p0]), cu_q=np.array([0, q1 - q0]),
                   cu_seg=np.array([0, len(segs)]))
        np.testing.assert_array_equal(out[q0:q1], oracle.packed_attn(one))


@pytest.mark.parametrize("bad", ["overlap", "gap", "shifted", "later_parent", "bidir_parent",
                                 "bidir_parent_alone", "long_parent", "nested", "len_without_parent",
                                 "empty_seg", "short_total", "bad_mode"])
def test_segment_checker_rejects(bad):
    segs = W.async_segments(4, 3, 2).astype(np.int64)
    N = int(segs[:, 1].sum())
    cu_q = [0, N]
    if bad == "overlap":
        segs[2, 0] -= 1
    elif bad == "gap":
        segs[2:, 0] += 1
        cu_q = [0, N + 1]
    elif bad == "shifted":  # a gap then an overlap: the lengths still add up
        segs[2, 0] += 1
    elif bad == "later_parent":
        segs[1, 3] = 2
    elif bad == "bidir_parent":
        segs[2, 3] = 1
    elif bad == "bidir_parent_alone":  # the parent has no parent but is not causal
        segs[1, 3], segs[1, 4] = -1, 0
        segs[2, 3], segs[2, 4] = 1, 1
    elif bad == "long_parent":
        segs[1, 4] = 5
    elif bad == "nested":
        segs[1, 2] = W.SEG_CAUSAL
        segs[2, 3] = 1
        segs[2, 4] = 1
    elif bad == "len_without_parent":
        segs[0, 4] = 1
    elif bad == "empty_seg":
        segs[3, 1] = 0
        segs[4:, 0] -= 4
        cu_q = [0, N - 4]
    elif bad == "short_total":
        cu_q = [0, N + 3]
    elif bad == "bad_mode":
        segs[1, 2] = 7
    assert oracle.check_segments(segs, cu_q, [0, len(segs)]) != 0


# ---------------------------------------------------------------- branch match
def _match_by_dict(inp):
    """Independent formulation: the first head index for each exact prefix tuple."""
    out = []
    for r in range(inp["heads"].shape[0]):
        table = {}
        for k in range(inp["heads"].shape[1]):
            n = int(inp["head_len"][r, k])
            table.setdefault(tuple(inp["heads"][r, k, :n].tolist()), k)
        v = tuple(inp["verified"][r, : int(inp["verified_len"][r])].tolist())
        out.append(table.get(v, -1))
    return np.array(out, np.int32)


def test_match_against_dict_lookup():
    inp = W.match_inputs(R=500, seed=71)
    got = oracle.branch_match(inp)
    np.testing.assert_array_equal(got, _match_by_dict(inp))
    hits = (got >= 0).mean()
    assert 0.5 < hits < 0.9


def test_match_tiny_alphabet_brute_force():
    # alphabet {0, 1}: many collisions, duplicate heads and ragged lengths
    rng = np.random.default_rng(72)
    R, M, B = 4000, 5, 3
    inp = dict(verified=rng.integers(0, 2, (R, B)).astype(np.int32),
               verified_len=rng.integers(0, B + 1, R).astype(np.int32),
               heads=rng.integers(0, 2, (R, M, B)).astype(np.int32),
               head_len=rng.integers(0, B + 1, (R, M)).astype(np.int32))
    got = oracle.branch_match(inp)
    np.testing.assert_array_equal(got, _match_by_dict(inp))
    assert (got == -1).any() and (got > 0).any()


def test_match_head0_never_hits_and_lowest_duplicate_wins():
    y = np.arange(1, 16, dtype=np.int32)[None]
    hb = W.branch_heads(y, 16, 12, 2, 1000, seed=1)
    heads, hl = hb["heads"], hb["head_len"]
    heads[0, 7] = heads[0, 3]
    hl[0, 7] = hl[0, 3]
    n = int(hl[0, 3])
    verified = np.zeros((1, 16), np.int32)
    verified[0, :n] = heads[0, 3, :n]
    got = oracle.branch_match(dict(verified=verified, verified_len=np.array([n], np.int32),
                                   heads=heads, head_len=hl))
    assert got[0] == 3
