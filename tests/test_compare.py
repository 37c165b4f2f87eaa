"""The parity rules of oracle/compare.py, checked on the CPU with outputs
planted from float64 arithmetic: an output the rules must accept (the
oracle's own, a flip of a decision that sits within the margin, a draw at
its CDF boundary) and outputs they must reject (a flip away from the
margin, a zero-weight token, a token two places from the boundary, wrong
padding)."""
import numpy as np
import pytest

import oracle
import workloads as W
from oracle import compare


def _inputs():
    return W.verify_inputs("cmp", 8, 3, 64, "f32", 77, family="sigma", sigmas=np.linspace(0.5, 3.0, 8),
                           delta=np.linspace(0.6, 1.4, 8))


def _run(x):
    return oracle.verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms)


def _report(x, o, tokens, accept_len):
    return compare.verify_report(tokens, accept_len, o["flags"].copy(), o, x.draft_ids, x.gamma, x.V, x.dtype, x=x)


def _cdf_draw(w, u):
    c = np.cumsum(w)
    return int(np.searchsorted(c, u * c[-1], side="right"))


def test_oracle_output_is_exact():
    x = _inputs()
    o = _run(x)
    rep = _report(x, o, o["tokens"].copy(), o["accept_len"].copy())
    assert rep["exact"] == x.B and rep["near_margin"] == 0 and not rep["mismatch"]
    assert rep["decisions"] == sum(min(int(n) + 1, x.gamma) + 1 for n in o["accept_len"])
    assert compare.near_margin_budget_ok(rep)


def _pick_rejectable(x):
    """A sequence whose first accept test has p/q < 1 (so a uniform can sit
    just on either side of it)."""
    for b in range(x.B):
        r = compare.accept_ratio(x, b, 0)
        if 0.05 < r < 0.95:
            return b, r
    raise AssertionError("no sequence with p/q < 1 at position 0")


def test_flip_within_margin_is_accepted_and_validated():
    x = _inputs()
    b, r = _pick_rejectable(x)
    x.uniforms[b, 0] = np.float32(r - 3e-6)  # the oracle accepts, 3e-6 from the margin
    assert x.uniforms[b, 0] < r and r - x.uniforms[b, 0] < compare.MARGIN
    o = _run(x)
    assert o["accept_len"][b] >= 1 and o["acc_margin"][b, 0] < compare.MARGIN
    # a GPU that rejected at position 0 draws from the residual of position 0
    w = compare.final_weights(x, b, 0)
    v = _cdf_draw(w, float(x.uniforms[b, x.gamma]))
    tok, n = o["tokens"].copy(), o["accept_len"].copy()
    tok[b] = -1
    tok[b, 0], n[b] = v, 0
    rep = _report(x, o, tok, n)
    assert rep["near_margin"] == 1 and not rep["mismatch"], rep
    # the same flip drawing a token of zero residual weight is invalid
    zero = np.nonzero(w == 0.0)[0]
    assert zero.size
    tok[b, 0] = int(zero[0])
    rep = _report(x, o, tok, n)
    assert rep["mismatch"] and "not a valid draw" in rep["mismatch"][0][1]
    # ... and so is one with bad padding
    tok[b, 0], tok[b, 2] = v, 5
    assert _report(x, o, tok, n)["mismatch"]


def test_flip_away_from_margin_is_a_mismatch():
    x = _inputs()
    o = _run(x)
    b = next(b for b in range(x.B) if np.all(o["acc_margin"][b, :min(o["accept_len"][b] + 1, x.gamma)] > 1e-3)
             and o["cdf_margin"][b] > 1e-3)
    tok, n = o["tokens"].copy(), o["accept_len"].copy()
    n_o = int(n[b])
    tok[b] = -1
    if n_o > 0:  # stop one test early: a decision far from its margin flipped
        w = compare.final_weights(x, b, n_o - 1)
        tok[b, :n_o - 1] = x.draft_ids[b, :n_o - 1]
        tok[b, n_o - 1], n[b] = _cdf_draw(w, float(x.uniforms[b, x.gamma])), n_o - 1
    else:
        tok[b, 0], n[b] = x.draft_ids[b, 0], 1
        tok[b, 1] = _cdf_draw(compare.final_weights(x, b, 1), float(x.uniforms[b, x.gamma]))
    rep = _report(x, o, tok, n)
    assert rep["mismatch"] and rep["near_margin"] == 0


def test_cdf_boundary_neighbour_only():
    """u * R within 1e-5 * R of a CDF breakpoint: the token on either side of
    it is valid, a token two places away is not."""
    x = _inputs()
    b, r = _pick_rejectable(x)
    x.uniforms[b, 0] = np.float32(min(0.999, r + 0.02))  # a clean rejection at position 0
    w = compare.final_weights(x, b, 0)
    pos = np.nonzero(w > 0.0)[0]
    assert pos.size >= 4
    c = np.cumsum(w)
    R = c[-1]
    k = pos[pos.size // 2]  # breakpoint C(k) between k and the next positive token
    u = np.float32(c[k] / R - 2e-6)
    x.uniforms[b, x.gamma] = u
    o = _run(x)
    assert o["accept_len"][b] == 0 and o["cdf_margin"][b] < compare.MARGIN
    nxt = pos[np.searchsorted(pos, k) + 1]
    for v, ok in ((k, True), (nxt, True), (pos[np.searchsorted(pos, k) + 2], False),
                  (pos[np.searchsorted(pos, k) - 1], False)):
        tok, n = o["tokens"].copy(), o["accept_len"].copy()
        tok[b, 0] = v
        rep = _report(x, o, tok, n)
        assert (not rep["mismatch"]) == ok, (v, k, rep)


def test_gumbel_validity_rule():
    """A Gumbel-max token is valid when its key is within the margin of the
    best key; the oracle's own token always is, a zero-weight one never."""
    x = _inputs()
    seed, offset = 99, 3
    o = oracle.gumbel_verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms, seed, offset)
    for b in range(x.B):
        n = int(o["accept_len"][b])
        w = compare.final_weights(x, b, n)
        assert compare.gumbel_token_ok(w, int(o["tokens"][b, n]), seed, offset, b, n)
        zero = np.nonzero(w == 0.0)[0]
        if zero.size:
            assert not compare.gumbel_token_ok(w, int(zero[0]), seed, offset, b, n)


def test_verify_report_requires_inputs():
    x = _inputs()
    o = _run(x)
    with pytest.raises(ValueError):
        compare.verify_report(o["tokens"], o["accept_len"], o["flags"], o, x.draft_ids, x.gamma, x.V, x.dtype)
