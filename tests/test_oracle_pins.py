"""Pins of the float64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a
library routine, a closed form, an invariant the pages state, a hand-derived
fixture, or an exact enumeration of the sampling law.  Page references:
"Breaking Entropy Bounds: Accelerating RL Training via MTP with Rejection
Sampling" (summary pages) and "EntMTP", Related Work "Speculative Decoding".
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=")
            vals[k.strip()] = [float(x) for x in v.split()]
    return vals


def _rows(rng, n, V, scale=1.5):
    return (rng.standard_normal((n, V)) * scale).astype(np.float64)


# ---------------------------------------------------------------- softmax --

@pytest.mark.parametrize("T", [0.6, 1.0, 1.7])
def test_softmax_matches_scipy(T):
    rng = np.random.default_rng(1)
    z = _rows(rng, 5, 1000, 3.0)
    ref = scipy.special.softmax(z / T, axis=-1)
    np.testing.assert_allclose(oracle.softmax(z, T), ref, rtol=1e-12, atol=1e-300)
    # log-probabilities against the library's log-sum-exp
    lse = scipy.special.logsumexp(z / T, axis=-1, keepdims=True)
    np.testing.assert_allclose(np.log(oracle.softmax(z, T)), z / T - lse, rtol=0, atol=1e-10)


def test_bf16_widening_is_exact():
    import torch

    x = np.random.default_rng(2).standard_normal((2, 64)).astype(np.float32) * 4
    b = torch.from_numpy(x).to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    ref = b.to(torch.float64).numpy()
    np.testing.assert_allclose(oracle.softmax(bits, 1.0), scipy.special.softmax(ref, axis=-1), rtol=1e-12)


# ------------------------------------------------------------ row stats ----

def test_alpha_equals_one_minus_tv():
    rng = np.random.default_rng(3)
    B, gamma, V = 6, 3, 777
    t = _rows(rng, B * (gamma + 1), V).reshape(B, gamma + 1, V)
    d = (t[:, :gamma] + rng.standard_normal((B, gamma, V)) * rng.uniform(0.05, 2.0, (B, 1, 1)))
    s = oracle.row_stats(t, d, np.full(B, 0.9))
    np.testing.assert_allclose(s["alpha"], 1.0 - s["tv"], rtol=0, atol=1e-12)
    assert np.all(s["alpha"] > 0) and np.all(s["alpha"] < 1)


def test_alpha_special_cases():
    rng = np.random.default_rng(4)
    V = 64
    z = _rows(rng, 2, V).reshape(1, 2, V)
    s = oracle.row_stats(z, z[:, :1].copy(), [1.3])
    assert abs(s["alpha"][0, 0] - 1.0) < 1e-14  # p == q
    # disjoint supports (-inf logits are zero probability)
    t = np.full((1, 2, V), -np.inf)
    d = np.full((1, 1, V), -np.inf)
    t[0, :, : V // 2] = 0.0
    d[0, 0, V // 2:] = 0.0
    s = oracle.row_stats(t, d, [1.0])
    assert s["alpha"][0, 0] == 0.0 and abs(s["tv"][0, 0] - 1.0) < 1e-15


def test_entropy_closed_forms():
    V = 1000
    uni = np.zeros((1, 2, V))
    s = oracle.row_stats(uni, uni[:, :1].copy(), [1.0])
    assert abs(s["entropy"][0, 0] - math.log(V)) < 1e-12
    onehot = np.full((1, 2, V), -np.inf)
    onehot[0, :, 17] = 3.0
    s = oracle.row_stats(onehot, onehot[:, :1].copy(), [0.7])
    assert s["entropy"][0, 0] == 0.0
    # library entropy and the target-only bound max p >= exp(-H) (summary App. D.2)
    rng = np.random.default_rng(5)
    z = _rows(rng, 4, V, 4.0).reshape(1, 4, V)
    s = oracle.row_stats(z, z[:, :3].copy(), [1.0])
    for i in range(4):
        p = scipy.special.softmax(z[0, i])
        assert abs(s["entropy"][0, i] - scipy.stats.entropy(p)) < 1e-12
        assert p.max() >= math.exp(-s["entropy"][0, i])


def test_proportional_mismatch_bound():
    """|q - p| <= delta p  =>  alpha >= 1 - delta/2 (summary App. D.4)."""
    rng = np.random.default_rng(6)
    V = 512
    for delta in (0.05, 0.3, 0.9):
        p = scipy.special.softmax(rng.standard_normal(V) * 2)
        # q = p (1 + delta s) with s in {-1, +1} chosen so sum p s = 0 exactly
        order = rng.permutation(V)
        half = order[: V // 2]
        s = np.ones(V)
        s[half] = -1.0
        w_plus, w_minus = p[s > 0].sum(), p[s < 0].sum()
        s[s > 0] *= min(1.0, w_minus / w_plus)
        s[s < 0] *= min(1.0, w_plus / w_minus)
        q = p * (1 + delta * s)
        assert np.all(np.abs(q - p) <= delta * p + 1e-15) and abs(q.sum() - 1) < 1e-12
        st = oracle.row_stats(np.log(np.stack([p, p]))[None], np.log(q)[None, None], [1.0])
        assert st["alpha"][0, 0] >= 1 - delta / 2 - 1e-12


# ------------------------------------------------------------ accept rule --

def _verify_rows(t_rows, d_rows, ids, us, T=1.0, want_stats=False):
    """Replicate one set of rows over a batch of (ids, uniforms)."""
    ids = np.asarray(ids, np.int32)
    us = np.asarray(us, np.float64)
    B = ids.shape[0]
    t = np.broadcast_to(t_rows, (B,) + t_rows.shape).copy()
    d = np.broadcast_to(d_rows, (B,) + d_rows.shape).copy()
    return oracle.verify(t, d, ids, np.full(B, T), us, want_stats)


def test_equal_rows_accept_everything():
    rng = np.random.default_rng(7)
    V, gamma = 300, 3
    t = _rows(rng, gamma + 1, V)
    d = t[:gamma].copy()
    us = [[0.0, 0.5, 0.999999, 0.2], [1 - 2.0 ** -24, 1 - 2.0 ** -24, 1 - 2.0 ** -24, 0.7]]
    ids = [[1, 2, 3], [299, 0, 150]]
    out = _verify_rows(t, d, ids, us)
    assert list(out["accept_len"]) == [3, 3]
    assert list(out["tokens"][0, :3]) == ids[0] and list(out["tokens"][1, :3]) == ids[1]


def test_one_hot_draft_accepts_with_probability_p():
    """q one-hot at y: accept iff u < p(y) (summary §2; App. D.2)."""
    rng = np.random.default_rng(8)
    V = 50
    t = _rows(rng, 2, V)
    y = 11
    d = np.full((1, V), -np.inf)
    d[0, y] = 0.0
    py = scipy.special.softmax(t[0])[y]
    out = _verify_rows(t, d, [[y], [y]], [[py * (1 - 1e-9), 0.5], [py * (1 + 1e-9), 0.5]])
    assert list(out["accept_len"]) == [1, 0]


def test_hand_fixture():
    g = _golden("hand_v3.txt")
    p, q = np.array(g["p"]), np.array(g["q"])
    t_rows = np.log(np.stack([p, p]))
    d_rows = np.log(q)[None]
    st = oracle.row_stats(t_rows[None], d_rows[None], [1.0])
    assert abs(st["alpha"][0, 0] - g["alpha"][0]) < 1e-15
    assert abs(st["tv"][0, 0] - g["tv"][0]) < 1e-15
    assert abs(st["entropy"][0, 0] - g["entropy"][0]) < 1e-15
    r = g["accept_ratio_y1"][0]
    out = _verify_rows(t_rows, d_rows, [[1], [1], [0], [0]],
                       [[r - 0.01, 0.5], [r + 0.01, 0.99], [0.999, 0.5], [0.0, 0.5]])
    assert list(out["accept_len"]) == [1, 0, 1, 1]
    assert out["tokens"][1, 0] == int(g["residual_token"][0])
    for u, tok in zip(g["bonus_u"], g["bonus_tokens"]):
        o = _verify_rows(t_rows, d_rows, [[0]], [[0.1, u]])
        assert o["tokens"][0, 1] == int(tok)
    tl = oracle.tv_loss(np.log(p)[None, None], np.log(q)[None, None], 1.0, 1.0)
    assert abs(tl["S"][0, 0] - g["S"][0]) < 1e-15
    assert abs(tl["loss"][0] + g["alpha"][0]) < 1e-15
    np.testing.assert_allclose(tl["grad"][0, 0], g["dloss_dz"], rtol=0, atol=1e-15)


def test_cdf_strict_breakpoint():
    """Smallest v with C(v) > u R: at u R == C(0) exactly the draw is v = 1."""
    t_rows = np.zeros((2, 2))  # p = (0.5, 0.5) exactly
    d_rows = np.zeros((1, 2))
    out = _verify_rows(t_rows, d_rows, [[0]], [[0.3, 0.5]])
    assert out["accept_len"][0] == 1 and out["tokens"][0, 1] == 1


# ----------------------------------------------- exact sampling-law checks --

def _intervals(weights):
    """u-intervals [a, b) over which the inverse CDF of `weights` is constant
    (breakpoints C(v)/R); returns (midpoints, lengths)."""
    w = np.maximum(weights, 0.0)
    c = np.concatenate([[0.0], np.cumsum(w) / w.sum()])
    a, b = c[:-1], c[1:]
    keep = b > a
    return (a[keep] + b[keep]) / 2, (b - a)[keep]


def _accept_regions(p, q, y):
    thr = min(1.0, p[y] / q[y]) if q[y] > 0 else 1.0
    regs = []
    if thr > 0:
        regs.append(("acc", thr / 2, thr))
    if thr < 1:
        regs.append(("rej", (thr + 1) / 2, 1 - thr))
    return regs


@pytest.mark.parametrize("T", [1.0, 0.8])
def test_enumeration_gamma1_law_is_p(T):
    """Output-token law equals p exactly (summary §2: RS preserves p; EntMTP
    "Speculative Decoding"): exhaustive enumeration at V = 8."""
    rng = np.random.default_rng(9)
    V = 8
    zt = _rows(rng, 2, V, 1.2)
    zd = zt[:1] + rng.standard_normal((1, V)) * 0.8
    p0, p1 = scipy.special.softmax(zt / T, axis=-1)
    q0 = scipy.special.softmax(zd[0] / T)
    cases, weights = [], []
    for y in range(V):
        for kind, u0, l0 in _accept_regions(p0, q0, y):
            w = p1 if kind == "acc" else np.maximum(p0 - q0, 0)
            for u1, l1 in zip(*_intervals(w)):
                cases.append((y, u0, u1))
                weights.append(q0[y] * l0 * l1)
    ids = [[c[0]] for c in cases]
    us = [[c[1], c[2]] for c in cases]
    out = _verify_rows(zt, zd, ids, us, T)
    weights = np.array(weights)
    first = np.zeros(V)
    second = np.zeros(V)
    np.add.at(first, out["tokens"][:, 0], weights)
    acc = out["accept_len"] == 1
    np.add.at(second, out["tokens"][acc, 1], weights[acc])
    np.testing.assert_allclose(first, p0, rtol=0, atol=1e-12)
    alpha = np.minimum(p0, q0).sum()
    np.testing.assert_allclose(weights[acc].sum(), alpha, atol=1e-12)
    np.testing.assert_allclose(second / alpha, p1, rtol=0, atol=1e-12)


def test_enumeration_gamma2_acceptance_product_and_tv_loss():
    """gamma = 2, fixed rows: P(n >= k) = prod_{i<=k} alpha_i, the second
    token given n >= 1 has law p_1, and E[n] equals minus the e2e TV loss of
    the same rows (summary §4: the loss is the expected acceptance length)."""
    rng = np.random.default_rng(10)
    V = 8
    zt = _rows(rng, 3, V, 1.0)
    zd = zt[:2] + rng.standard_normal((2, V)) * 0.7
    p = scipy.special.softmax(zt, axis=-1)
    q = scipy.special.softmax(zd, axis=-1)
    cases, weights = [], []
    for y0 in range(V):
        for k0, u0, l0 in _accept_regions(p[0], q[0], y0):
            if k0 == "rej":
                for u2, l2 in zip(*_intervals(np.maximum(p[0] - q[0], 0))):
                    cases.append(([y0, 0], [u0, 0.5, u2]))
                    weights.append(q[0][y0] * l0 * l2)
                continue
            for y1 in range(V):
                for k1, u1, l1 in _accept_regions(p[1], q[1], y1):
                    w = p[2] if k1 == "acc" else np.maximum(p[1] - q[1], 0)
                    for u2, l2 in zip(*_intervals(w)):
                        cases.append(([y0, y1], [u0, u1, u2]))
                        weights.append(q[0][y0] * l0 * q[1][y1] * l1 * l2)
    out = _verify_rows(zt, zd, [c[0] for c in cases], [c[1] for c in cases])
    w = np.array(weights)
    n = out["accept_len"]
    a = np.minimum(p[:2], q).sum(axis=1)
    assert abs(w.sum() - 1) < 1e-12
    assert abs(w[n >= 1].sum() - a[0]) < 1e-12
    assert abs(w[n >= 2].sum() - a[0] * a[1]) < 1e-12
    first = np.zeros(V)
    np.add.at(first, out["tokens"][:, 0], w)
    np.testing.assert_allclose(first, p[0], atol=1e-12)
    second = np.zeros(V)
    m = n >= 1
    np.add.at(second, out["tokens"][m, 1], w[m])
    np.testing.assert_allclose(second / a[0], p[1], atol=1e-12)
    third = np.zeros(V)
    m = n >= 2
    np.add.at(third, out["tokens"][m, 2], w[m])
    np.testing.assert_allclose(third / (a[0] * a[1]), p[2], atol=1e-12)
    tl = oracle.tv_loss(zt[None, :2], zd[None], 1.0, 1.0, with_grad=False)
    assert abs(-tl["loss"][0] - (w * n).sum()) < 1e-12


# --------------------------------------------------------- TV loss / grad --

def _kink_free_inputs(rng, N, gamma, V, T, min_gap=1e-3):
    while True:
        t = rng.standard_normal((N, gamma, V)) * 1.3
        d = t + rng.standard_normal((N, gamma, V)) * 0.6
        p = scipy.special.softmax(t / T, axis=-1)
        q = scipy.special.softmax(d / T, axis=-1)
        if np.abs(p - q).min() > min_gap:
            return t, d


@pytest.mark.parametrize("T,scale", [(1.0, 1.0), (0.7, 2.5)])
def test_tv_gradient_finite_differences(T, scale):
    """Analytic gradient (summary App. A, chained through the product of
    §4) against central differences of the loss, h = 1e-6."""
    rng = np.random.default_rng(11)
    N, gamma, V = 2, 3, 16
    t, d = _kink_free_inputs(rng, N, gamma, V, T, 2e-4)
    out = oracle.tv_loss(t, d, T, scale)
    h = 1e-6
    fd = np.empty_like(d)
    for idx in np.ndindex(d.shape):
        dp = d.copy()
        dm = d.copy()
        dp[idx] += h
        dm[idx] -= h
        lp = oracle.tv_loss(t, dp, T, 1.0, with_grad=False)["loss"].sum()
        lm = oracle.tv_loss(t, dm, T, 1.0, with_grad=False)["loss"].sum()
        fd[idx] = scale * (lp - lm) / (2 * h)
    np.testing.assert_allclose(out["grad"], fd, rtol=0, atol=1e-7)


def test_tv_gradient_structure():
    """sum_j dalpha/dz_j = 0 and |dalpha/dz_j| <= q_j / T (App. A bound)."""
    rng = np.random.default_rng(12)
    N, gamma, V, T = 3, 3, 200, 0.8
    t = rng.standard_normal((N, gamma, V)) * 2
    d = t + rng.standard_normal((N, gamma, V)) * 0.5
    out = oracle.tv_loss(t, d, T, 1.0)
    q = scipy.special.softmax(d / T, axis=-1)
    dadz = out["grad"] / out["g"][:, :, None]
    assert np.abs(dadz.sum(-1)).max() < 1e-15
    assert np.all(np.abs(dadz) <= q / T + 1e-15)
    assert np.all((out["S"] >= 0) & (out["S"] <= 1))


def test_e2e_loss_special_cases():
    rng = np.random.default_rng(13)
    V = 100
    # gamma = 1: l = -alpha
    t = rng.standard_normal((4, 1, V))
    d = t + rng.standard_normal((4, 1, V))
    out = oracle.tv_loss(t, d, 1.0, 1.0, with_grad=False)
    np.testing.assert_allclose(out["loss"], -out["alpha"][:, 0], atol=0)
    # all alpha = 1 (p == q): l = -gamma, gradient zero under either tie rule
    t = rng.standard_normal((2, 5, V))
    for tie in (True, False):
        out = oracle.tv_loss(t, t.copy(), 1.0, 1.0, tie_le=tie)
        np.testing.assert_allclose(out["loss"], -5.0, atol=1e-12)
        assert np.abs(out["grad"]).max() < 1e-15
    # alpha_0 = 0 zeroes every term; g_0 = -(1 + alpha_1 + alpha_1 alpha_2) = -3, later g_k = 0
    t = np.full((1, 3, V), -np.inf)
    d = np.full((1, 3, V), -np.inf)
    t[0, 0, :50] = 0
    d[0, 0, 50:] = 0
    t[0, 1:] = 0
    d[0, 1:] = 0
    out = oracle.tv_loss(t, d, 1.0, 1.0)
    assert out["loss"][0] == 0.0 and abs(out["g"][0, 0] + 3.0) < 1e-12 and np.all(out["g"][0, 1:] == 0)
    assert np.isfinite(out["grad"]).all()


# ----------------------------------------------------------------- flags ---

def test_flags_and_defined_outputs():
    rng = np.random.default_rng(14)
    B, gamma, V = 6, 2, 40
    t = rng.standard_normal((B, gamma + 1, V))
    d = t[:, :gamma] + 0.1
    ids = np.zeros((B, gamma), np.int32)
    u = np.full((B, gamma + 1), 0.5)
    temp = np.ones(B)
    temp[1] = -1.0  # T = 0 is greedy decoding, a negative temperature is invalid
    ids[2, 1] = V
    u[3, 0] = 1.0
    t[4, 0, 7] = np.nan
    d[5, 0, :] = -np.inf
    out = oracle.verify(t, d, ids, temp, u)
    assert out["flags"][0] == 0 and out["accept_len"][0] >= 0
    assert out["flags"][1] == oracle.ROW_BAD_TEMP
    assert out["flags"][2] == oracle.ROW_BAD_ID
    assert out["flags"][3] == oracle.ROW_BAD_UNIFORM
    assert out["flags"][4] == oracle.ROW_NONFINITE
    assert out["flags"][5] == oracle.ROW_NONFINITE
    for b in range(1, B):
        assert out["accept_len"][b] == -1 and np.all(out["tokens"][b] == -1)


# ------------------------------------------------ greedy and target-only --

def _greedy_reference(t, ids):
    """Greedy decoding written out with numpy arg max (first index among
    equals): accept while the draft is the target's arg max, then emit it."""
    toks = []
    for i in range(ids.shape[0] + 1):
        a = int(np.argmax(t[i]))
        if i < ids.shape[0] and ids[i] == a:
            toks.append(a)
            continue
        toks.append(a)
        break
    n = len(toks) - 1
    return toks + [-1] * (ids.shape[0] + 1 - len(toks)), n


def test_greedy_verify_is_the_argmax_prefix():
    """T = 0 is greedy decoding: p and q one-hot at their arg max, so rejection
    sampling accepts a draft iff it is the target's arg max (summary App. D.2,
    App. G: target-only selects by arg max)."""
    rng = np.random.default_rng(21)
    B, gamma, V = 40, 4, 60
    t = rng.standard_normal((B, gamma + 1, V))
    t[5, 2, 7] = t[5, 2].max() + 1.0
    t[5, 2, 3] = t[5, 2, 7]  # a tie: the smaller index wins
    ids = np.where(rng.random((B, gamma)) < 0.7, t[:, :gamma].argmax(-1), rng.integers(0, V, (B, gamma))).astype(np.int32)
    d = rng.standard_normal((B, gamma, V))
    u = rng.random((B, gamma + 1))
    out = oracle.verify(t, d, ids, np.zeros(B), u)
    to = oracle.to_verify(t, np.where(np.arange(V)[None, None] == ids[..., None], 5.0, 0.0), np.zeros(B), u)
    for b in range(B):
        toks, n = _greedy_reference(t[b], ids[b])
        assert list(out["tokens"][b]) == toks and out["accept_len"][b] == n, b
        assert list(to["tokens"][b]) == toks and to["accept_len"][b] == n, b
    assert np.all(out["flags"] == 0)
    # statistics need T > 0
    assert np.all(oracle.verify(t[:2], d[:2], ids[:2], np.zeros(2), u[:2], want_stats=True)["flags"] == oracle.ROW_BAD_TEMP)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_target_only_law_is_p_enumeration(T):
    """Target-only sampling (summary §2, App. D.2): the draft is arg max q,
    accepted with probability p(yhat); the replacement at a rejection is drawn
    from p without yhat.  Exhaustive enumeration at V = 8: the first-token law
    is p exactly and the acceptance probability is p(yhat)."""
    rng = np.random.default_rng(22)
    V = 8
    zt = _rows(rng, 2, V, 1.3)
    zd = zt[:1] + rng.standard_normal((1, V)) * 0.9
    p0, p1 = scipy.special.softmax(zt / T, axis=-1)
    yhat = int(np.argmax(zd[0]))
    py = p0[yhat]
    resid = p0.copy()
    resid[yhat] = 0.0
    cases, weights, kinds = [], [], []
    for kind, u0, l0 in [("acc", py / 2, py), ("rej", (py + 1) / 2, 1 - py)]:
        w = p1 if kind == "acc" else resid
        for u1, l1 in zip(*_intervals(w)):
            cases.append([u0, u1])
            weights.append(l0 * l1)
            kinds.append(kind)
    B = len(cases)
    out = oracle.to_verify(np.broadcast_to(zt, (B, 2, V)).copy(), np.broadcast_to(zd, (B, 1, V)).copy(),
                           np.full(B, T), np.array(cases))
    weights = np.array(weights)
    assert np.all(out["yhat"][:, 0] == yhat)
    first = np.zeros(V)
    np.add.at(first, out["tokens"][:, 0], weights)
    np.testing.assert_allclose(first, p0, rtol=0, atol=1e-12)
    acc = out["accept_len"] == 1
    np.testing.assert_allclose(weights[acc].sum(), py, atol=1e-12)
    second = np.zeros(V)
    np.add.at(second, out["tokens"][acc, 1], weights[acc])
    np.testing.assert_allclose(second / py, p1, rtol=0, atol=1e-12)


def test_target_only_acceptance_product():
    """gamma = 2: P(n >= 1) = p_0(yhat_0) and P(n >= 2) = p_0(yhat_0) p_1(yhat_1)."""
    rng = np.random.default_rng(23)
    V = 8
    zt = _rows(rng, 3, V, 1.0)
    zd = zt[:2] + rng.standard_normal((2, V)) * 0.7
    p = scipy.special.softmax(zt, axis=-1)
    y = zd.argmax(-1)
    a0, a1 = p[0, y[0]], p[1, y[1]]
    cases, weights = [], []
    for u0, l0 in [(a0 / 2, a0), ((a0 + 1) / 2, 1 - a0)]:
        for u1, l1 in [(a1 / 2, a1), ((a1 + 1) / 2, 1 - a1)]:
            cases.append([u0, u1, 0.5])
            weights.append(l0 * l1)
    B = len(cases)
    out = oracle.to_verify(np.broadcast_to(zt, (B, 3, V)).copy(), np.broadcast_to(zd, (B, 2, V)).copy(),
                           np.ones(B), np.array(cases))
    n = out["accept_len"]
    w = np.array(weights)
    np.testing.assert_allclose(w[n >= 1].sum(), a0, atol=1e-12)
    np.testing.assert_allclose(w[n >= 2].sum(), a0 * a1, atol=1e-12)


def test_diagnostics_against_library_routines():
    """alpha = 1 - TV; H(q) and D_KL(q || p) as scipy.stats.entropy computes
    them; yhat = arg max q; p(yhat); rs_better = [TV < 1 - p(yhat)]
    (summary App. E)."""
    rng = np.random.default_rng(24)
    B, gamma, V = 6, 3, 400
    t = rng.standard_normal((B, gamma + 1, V)) * np.linspace(0.5, 4, B)[:, None, None]
    d = t[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.6
    T = np.linspace(0.6, 1.4, B)
    o = oracle.diagnostics(t, d, T)
    assert np.all(o["flags"] == 0)
    for b in range(B):
        for i in range(gamma):
            p = scipy.special.softmax(t[b, i] / T[b])
            q = scipy.special.softmax(d[b, i] / T[b])
            assert o["yhat"][b, i] == int(np.argmax(q))
            np.testing.assert_allclose(o["ent_q"][b, i], scipy.stats.entropy(q), rtol=1e-12)
            np.testing.assert_allclose(o["kl"][b, i], scipy.stats.entropy(q, p), rtol=1e-10)
            np.testing.assert_allclose(o["p_yhat"][b, i], p[np.argmax(q)], rtol=1e-12)
            tv = 0.5 * np.abs(p - q).sum()
            np.testing.assert_allclose(o["alpha"][b, i], 1 - tv, atol=1e-12)
            assert o["rs_better"][b, i] == int(tv < 1 - p[np.argmax(q)])
        for i in range(gamma + 1):
            np.testing.assert_allclose(o["ent_p"][b, i], scipy.stats.entropy(scipy.special.softmax(t[b, i] / T[b])),
                                       rtol=1e-12)
    # D_KL(q || q) = 0, and an unsupported q mass makes it infinite
    same = oracle.diagnostics(t[:1], t[:1, :gamma], [1.0])
    np.testing.assert_allclose(same["kl"], 0.0, atol=1e-12)
    masked = t[:1].copy()
    masked[0, 0, 0] = -np.inf
    assert np.isinf(oracle.diagnostics(masked, t[:1, :gamma], [1.0])["kl"][0, 0])


def test_decision_boundary_matches_enumerated_acceptance():
    """Summary App. E: rejection sampling accepts the first draft more often
    than target-only sampling iff d_TV(p, q) < 1 - p(yhat).  The acceptance
    probabilities are enumerated from the two verify oracles (y ~ q with the
    accept threshold of each draft, and the target-only threshold)."""
    rng = np.random.default_rng(25)
    V = 8
    seen = set()
    for trial in range(40):
        zt = _rows(rng, 2, V, rng.uniform(0.3, 3.0))
        zd = zt[:1] + rng.standard_normal((1, V)) * rng.uniform(0.05, 2.5)
        p0 = scipy.special.softmax(zt[0])
        q0 = scipy.special.softmax(zd[0])
        # RS: y ~ q, accept region of u per y
        ids, us, w = [], [], []
        for y in range(V):
            for kind, u0, l0 in _accept_regions(p0, q0, y):
                ids.append([y])
                us.append([u0, 0.5])
                w.append(q0[y] * l0)
        rs = _verify_rows(zt, zd, ids, us)
        p_rs = np.array(w)[rs["accept_len"] == 1].sum()
        # TO: one draft (arg max q), two u-regions
        py = p0[np.argmax(zd[0])]
        to = oracle.to_verify(np.broadcast_to(zt, (2, 2, V)).copy(), np.broadcast_to(zd, (2, 1, V)).copy(),
                              np.ones(2), np.array([[py / 2, 0.5], [(py + 1) / 2, 0.5]]))
        p_to = np.array([py, 1 - py])[to["accept_len"] == 1].sum()
        dg = oracle.diagnostics(zt[None], zd[None], [1.0])
        if dg["boundary_margin"][0, 0] < 1e-9:
            continue
        assert dg["rs_better"][0, 0] == int(p_rs > p_to), trial
        seen.add(int(p_rs > p_to))
    assert seen == {0, 1}


# ------------------------------------------------ Gumbel-max final draw ----

def _kat(name):
    rows = []
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(w, 16) for w in line.split()])
    return rows


def test_philox_known_answers():
    """The oracle's Philox4x32-10 reproduces the generator's published
    known-answer vectors (tests/golden/philox4x32_10_kat.txt)."""
    rows = _kat("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        out = oracle.philox4x32_10(r[0:4], r[4:6])
        assert [int(x) for x in out] == r[6:10]


def test_gumbel_noise_is_standard_gumbel():
    """G_v = -ln(-ln U_v) from the Philox stream is standard Gumbel: a
    Kolmogorov-Smirnov test against the library Gumbel law, the mean (Euler's
    constant) and the variance (pi^2 / 6); distinct rows, sequences, offsets
    and seeds give distinct streams."""
    g = np.concatenate([oracle.gumbel_noise(7, 0, b, i, 0, 4000) for b in range(5) for i in range(5)])
    assert scipy.stats.kstest(g, scipy.stats.gumbel_r.cdf).pvalue > 1e-3
    assert abs(g.mean() - np.euler_gamma) < 0.02
    assert abs(g.var() - math.pi ** 2 / 6) < 0.05
    a = oracle.gumbel_noise(7, 0, 0, 0, 0, 64)
    for other in (oracle.gumbel_noise(7, 0, 1, 0, 0, 64), oracle.gumbel_noise(7, 0, 0, 1, 0, 64),
                  oracle.gumbel_noise(7, 1, 0, 0, 0, 64), oracle.gumbel_noise(8, 0, 0, 0, 0, 64),
                  oracle.gumbel_noise(7 + (1 << 32), 0, 0, 0, 0, 64)):
        assert not np.any(a == other)
    # word v mod 4 of counter v / 4: v = 0..3 share one counter
    np.testing.assert_array_equal(oracle.gumbel_noise(7, 0, 0, 0, 2, 6), a[2:8])


def _chi2_ok(counts, probs, q=0.999):
    keep = probs > 0
    assert counts[~keep].sum() == 0
    n = counts.sum()
    e = n * probs[keep]
    chi2 = ((counts[keep] - e) ** 2 / e).sum()
    return chi2 < scipy.stats.chi2.ppf(q, keep.sum() - 1), chi2


def test_gumbel_final_draw_law():
    """The Gumbel-max final draw (summary App. G.2) samples the residual
    norm(max(0, p - q)) at a certain rejection and p_gamma after gamma
    accepts: chi-square over 30,000 independent streams (one per sequence)
    at V = 8, with every accept decision the same."""
    V, B = 8, 30000
    rng = np.random.default_rng(31)
    zt = rng.standard_normal((2, V)) * 1.2
    zd = rng.standard_normal(V) * 1.2
    p0, p1 = scipy.special.softmax(zt, axis=1)
    q0 = scipy.special.softmax(zd)
    # rejection at position 0: the draft token where q is largest relative to p, u close to 1
    y = int(np.argmax(q0 / p0))
    t = np.broadcast_to(zt, (B, 2, V)).copy()
    d = np.broadcast_to(zd, (B, 1, V)).copy()
    ids = np.full((B, 1), y, np.int32)
    u = np.tile([[0.9999, 0.5]], (B, 1))
    out = oracle.gumbel_verify(t, d, ids, np.ones(B), u, seed=1234, offset=3)
    assert np.all(out["accept_len"] == 0) and np.all(out["flags"] == 0)
    r = np.maximum(p0 - q0, 0)
    ok, chi2 = _chi2_ok(np.bincount(out["tokens"][:, 0], minlength=V), r / r.sum())
    assert ok, chi2
    # all accepted (q == p): the bonus token follows p_1
    d2 = np.broadcast_to(zt[0], (B, 1, V)).copy()
    out = oracle.gumbel_verify(t, d2, ids, np.ones(B), u, seed=99)
    assert np.all(out["accept_len"] == 1)
    ok, chi2 = _chi2_ok(np.bincount(out["tokens"][:, 1], minlength=V), p1)
    assert ok, chi2


def test_gumbel_verify_acceptance_is_the_rejection_sampling_chain():
    """Only the final draw changes: accept lengths, accepted tokens and flags
    equal those of the inverse-CDF verify, greedy rows (T = 0) entirely;
    u[b, gamma] is not examined."""
    rng = np.random.default_rng(32)
    B, gamma, V = 64, 4, 200
    t = rng.standard_normal((B, gamma + 1, V)) * 2
    d = t[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.7
    ids = rng.integers(0, V, (B, gamma)).astype(np.int32)
    T = np.where(np.arange(B) % 5 == 0, 0.0, rng.uniform(0.6, 1.4, B))
    u = rng.random((B, gamma + 1))
    a = oracle.verify(t, d, ids, T, u)
    u2 = u.copy()
    u2[:, gamma] = 7.0  # not a valid uniform, and not used by the Gumbel draw
    g = oracle.gumbel_verify(t, d, ids, T, u2, seed=5)
    np.testing.assert_array_equal(a["accept_len"], g["accept_len"])
    np.testing.assert_array_equal(a["flags"], g["flags"])
    for b in range(B):
        n = a["accept_len"][b]
        np.testing.assert_array_equal(a["tokens"][b, :n], g["tokens"][b, :n])
        if T[b] == 0:
            np.testing.assert_array_equal(a["tokens"][b], g["tokens"][b])
    assert (a["accept_len"] < gamma).any() and (a["accept_len"] == gamma).any()
    # the draw depends on the stream: another seed changes some final tokens
    g2 = oracle.gumbel_verify(t, d, ids, T, u2, seed=6)
    fin = np.array([g["tokens"][b, g["accept_len"][b]] for b in range(B)])
    fin2 = np.array([g2["tokens"][b, g2["accept_len"][b]] for b in range(B)])
    assert (fin != fin2).any()


# -------------------------------------------- TV-loss layout and variants --

def test_shared_target_layout_is_the_row_gather():
    """Shared target rows [N + gamma - 1, V]: pair (t, k) uses row t + k, the
    target distribution at the token draft step k of position t predicts.
    Equal to the per-position loss on the explicitly gathered target."""
    rng = np.random.default_rng(41)
    N, gamma, V = 7, 3, 50
    ts = rng.standard_normal((N + gamma - 1, V)) * 2
    d = rng.standard_normal((N, gamma, V)) * 2
    gathered = np.stack([np.stack([ts[t + k] for k in range(gamma)]) for t in range(N)])
    a = oracle.tv_loss(gathered, d, 0.9, 1.5)
    b = oracle.tv_loss(ts, d, 0.9, 1.5, shared_target=True)
    for key in ("loss", "alpha", "S", "g", "grad"):
        np.testing.assert_array_equal(a[key], b[key])
    c = oracle.tv_loss(ts, d, 0.9, 1.5, shared_target=True, clamp_tau=0.4)
    e = oracle.tv_loss(gathered, d, 0.9, 1.5, clamp_tau=0.4)
    for key in ("loss", "alpha", "grad"):
        np.testing.assert_array_equal(c[key], e[key])


def test_clamped_step_loss_closed_forms():
    """App. F per-step loss clamp(1 - alpha, 0, tau_max): with tau_max >= 1 it
    is the summed total variation 1/2 sum |p - q| (a library softmax), with
    tau_max = 0 it vanishes with a zero gradient, and a step whose 1 - alpha
    exceeds tau_max contributes tau_max and no gradient."""
    rng = np.random.default_rng(42)
    N, gamma, V, T = 5, 3, 80, 1.1
    t = rng.standard_normal((N, gamma, V)) * 2
    d = t + rng.standard_normal((N, gamma, V)) * 0.8
    p = scipy.special.softmax(t / T, axis=-1)
    q = scipy.special.softmax(d / T, axis=-1)
    tv = 0.5 * np.abs(p - q).sum(-1)
    out = oracle.tv_loss(t, d, T, 1.0, clamp_tau=1.0)
    np.testing.assert_allclose(out["loss"], tv.sum(-1), rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(out["g"], -1.0)
    z = oracle.tv_loss(t, d, T, 1.0, clamp_tau=0.0)
    assert np.all(z["loss"] == 0) and np.all(z["grad"] == 0)
    tau = float(np.median(tv))
    c = oracle.tv_loss(t, d, T, 1.0, clamp_tau=tau)
    np.testing.assert_allclose(c["loss"], np.minimum(tv, tau).sum(-1), rtol=1e-12, atol=1e-14)
    over = tv > tau
    assert over.any() and (~over).any()
    assert np.all(c["grad"][over] == 0)
    # inside the clamp: the gradient of -alpha, i.e. that of the e2e loss at gamma = 1
    one = oracle.tv_loss(t[:, :1], d[:, :1], T, 1.0)
    inside = ~over[:, 0]
    np.testing.assert_allclose(c["grad"][inside, 0], one["grad"][inside, 0], rtol=0, atol=1e-15)


def test_clamped_step_loss_finite_differences():
    """Gradient of sum_k clamp(1 - alpha_k, 0, tau_max) against central
    differences, with tau_max between the steps' 1 - alpha so that both the
    clamped and the open side occur and no step sits on a kink."""
    rng = np.random.default_rng(43)
    N, gamma, V, T = 2, 3, 12, 0.9
    t, d = _kink_free_inputs(rng, N, gamma, V, T, 2e-4)
    a = oracle.tv_loss(t, d, T, 1.0)["alpha"]
    steps = np.sort((1 - a).ravel())
    tau = 0.5 * (steps[2] + steps[3])
    assert np.min(np.abs((1 - a) - tau)) > 1e-3
    out = oracle.tv_loss(t, d, T, 2.0, clamp_tau=tau)
    h = 1e-6
    fd = np.empty_like(d)
    for idx in np.ndindex(d.shape):
        dp = d.copy()
        dm = d.copy()
        dp[idx] += h
        dm[idx] -= h
        lp = oracle.tv_loss(t, dp, T, 1.0, with_grad=False, clamp_tau=tau)["loss"].sum()
        lm = oracle.tv_loss(t, dm, T, 1.0, with_grad=False, clamp_tau=tau)["loss"].sum()
        fd[idx] = 2.0 * (lp - lm) / (2 * h)
    np.testing.assert_allclose(out["grad"], fd, rtol=0, atol=1e-7)
    assert (out["g"] == 0).any() and (out["g"] == -1).any()


# ---------------------------------------------------------- draft sampling --

@pytest.mark.parametrize("T", [1.0, 0.6])
def test_draft_sample_multinomial_law_enumeration(T):
    """Multinomial draft sampling (summary App. G.1, the draft stage draws
    from q): the inverse-CDF draw is piecewise constant in u with
    breakpoints C(v) / R; evaluating at every interval midpoint, weighted by
    the interval length, gives softmax(z / T) (a library routine) to 1e-12."""
    rng = np.random.default_rng(51)
    V = 8
    z = rng.standard_normal(V) * 1.5
    q = scipy.special.softmax(z / T)
    edges = np.concatenate([[0.0], np.cumsum(q)])
    edges[-1] = 1.0
    mids = 0.5 * (edges[:-1] + edges[1:])
    out = oracle.draft_sample(np.tile(z, (V, 1)), np.full(V, T), mids)
    law = np.zeros(V)
    for i, tok in enumerate(out["ids"]):
        law[tok] += edges[i + 1] - edges[i]
    np.testing.assert_allclose(law, q, rtol=0, atol=1e-12)
    assert np.all(out["flags"] == 0)


def test_draft_sample_hand_fixture_and_greedy():
    """The V = 3 bonus-draw fixture (C = (0.5, 0.8, 1.0)) applies to the draft
    draw; T = 0 is the arg max with ties to the smaller index; bad
    temperature and uniform are flagged."""
    z = np.log(np.array([[0.5, 0.3, 0.2]] * 3))
    out = oracle.draft_sample(z, np.ones(3), np.array([0.3, 0.79, 0.81]))
    assert list(out["ids"]) == [0, 1, 2]
    zz = np.array([[1.0, 3.0, 3.0, -1.0], [0.0, 0.0, 0.0, 0.0]])
    g = oracle.draft_sample(zz, np.zeros(2), np.array([0.5, 0.5]))
    assert list(g["ids"]) == [1, 0] and np.all(g["flags"] == 0)
    # greedy rows draw nothing, but their uniform is still checked (as in verification)
    assert list(oracle.draft_sample(zz, np.zeros(2), np.array([7.0, 0.5]))["flags"]) == [oracle.ROW_BAD_UNIFORM, 0]
    bad = oracle.draft_sample(zz, np.array([-1.0, 1.0]), np.array([0.5, 1.0]))
    assert list(bad["flags"]) == [oracle.ROW_BAD_TEMP, oracle.ROW_BAD_UNIFORM] and list(bad["ids"]) == [-1, -1]


def test_draft_sample_gumbel_law():
    """Gumbel-max draft sampling (summary App. G.2, vLLM): chi-square of
    30,000 rows with independent streams against softmax(z / T)."""
    V, R, T = 8, 30000, 0.8
    z = np.random.default_rng(52).standard_normal(V) * 1.3
    out = oracle.draft_sample(np.tile(z, (R, 1)), np.full(R, T), method="gumbel", seed=77, offset=5)
    ok, chi2 = _chi2_ok(np.bincount(out["ids"], minlength=V), scipy.special.softmax(z / T))
    assert ok, chi2
    # the draw is the arg max of ln q + G over the row's own noise stream
    g = oracle.gumbel_noise(77, 5, 3, 0, 0, V)
    assert out["ids"][3] == int(np.argmax(np.log(scipy.special.softmax(z / T)) + g))


# ----------------------------------------------------------- top-K TV path --

def _topk(t, K):
    idx = np.argsort(-t, axis=-1, kind="stable")[..., :K].astype(np.int32)
    return np.take_along_axis(t, idx, axis=-1), idx


def test_topk_with_every_entry_is_the_full_loss():
    """K = V (a shuffled full list): the top-K loss, alpha, S and gradient
    equal the full TV loss (App. F top-K path, K = |V|)."""
    rng = np.random.default_rng(61)
    N, gamma, V = 3, 3, 40
    t = rng.standard_normal((N, gamma, V)) * 2
    d = t + rng.standard_normal((N, gamma, V)) * 0.6
    perm = np.stack([np.stack([rng.permutation(V) for _ in range(gamma)]) for _ in range(N)]).astype(np.int32)
    vals = np.take_along_axis(t, perm, axis=-1)
    a = oracle.tv_loss(t, d, 0.8, 1.5)
    b = oracle.tv_loss_topk(vals, perm, d, 0.8, 1.5)
    for key in ("loss", "alpha", "S", "g", "grad"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-12, atol=1e-14)


def test_topk_is_the_loss_against_the_truncated_target():
    """The top-K target is the softmax renormalised over its K entries: the
    same as the full loss with every other target logit at -inf (p = 0), a
    different code path of the oracle; also for the clamped loss."""
    rng = np.random.default_rng(62)
    N, gamma, V, K = 4, 3, 64, 9
    t = rng.standard_normal((N, gamma, V)) * 2.5
    d = t + rng.standard_normal((N, gamma, V)) * 0.7
    vals, idx = _topk(t, K)
    masked = np.full_like(t, -np.inf)
    np.put_along_axis(masked, idx, vals, axis=-1)
    for tau in (None, 0.5):
        a = oracle.tv_loss(masked, d, 1.1, 2.0, clamp_tau=tau)
        b = oracle.tv_loss_topk(vals, idx, d, 1.1, 2.0, clamp_tau=tau)
        for key in ("loss", "alpha", "S", "g", "grad"):
            np.testing.assert_allclose(b[key], a[key], rtol=1e-12, atol=1e-14)
    # alpha~ <= 1 and it shrinks with K (less target mass overlaps q)
    a_small = oracle.tv_loss_topk(*_topk(t, 2), d, 1.1, with_grad=False)["alpha"]
    assert np.all(a_small <= 1) and np.mean(a_small) < np.mean(oracle.tv_loss_topk(vals, idx, d, 1.1)["alpha"])


def test_topk_gradient_finite_differences():
    """Gradient w.r.t. the draft logits against central differences."""
    rng = np.random.default_rng(63)
    N, gamma, V, K, T = 2, 3, 14, 5, 0.9
    while True:
        t = rng.standard_normal((N, gamma, V)) * 1.5
        d = t + rng.standard_normal((N, gamma, V)) * 0.6
        vals, idx = _topk(t, K)
        pk = scipy.special.softmax(vals / T, axis=-1)
        q = scipy.special.softmax(d / T, axis=-1)
        if np.abs(np.take_along_axis(q, idx, axis=-1) - pk).min() > 2e-4:
            break
    out = oracle.tv_loss_topk(vals, idx, d, T, 1.5)
    h = 1e-6
    fd = np.empty_like(d)
    for ix in np.ndindex(d.shape):
        dp = d.copy()
        dm = d.copy()
        dp[ix] += h
        dm[ix] -= h
        lp = oracle.tv_loss_topk(vals, idx, dp, T, 1.0, with_grad=False)["loss"].sum()
        lm = oracle.tv_loss_topk(vals, idx, dm, T, 1.0, with_grad=False)["loss"].sum()
        fd[ix] = 1.5 * (lp - lm) / (2 * h)
    np.testing.assert_allclose(out["grad"], fd, rtol=0, atol=1e-7)
    assert oracle.tv_loss_topk(vals, np.where(idx == idx[0, 0, 0], V, idx), d, T)["flags"][0] == oracle.ROW_BAD_ID
