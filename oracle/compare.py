"""Parity checks of library outputs against the float64 oracle (test
infrastructure, used by the test suite and the smoke check).

Rules (tolerances fixed by the method's accuracy bar):
* token ids and accept lengths must be identical, except in sequences where
  a decision the oracle took is near its margin: |u_i - p_i(y)/q_i(y)| <
  1e-5 for an accept test, or a CDF margin below 1e-5 for the final draw.
  Those sequences are counted (they must stay below 1 % of the decisions
  on the full-size workloads) and checked for validity against float64
  weights from the inputs: the flipped decision is the near one, the
  accepted prefix equals the draft ids, and the drawn token has positive
  weight and is the draw at the uniform up to the margin (the oracle's
  token or its neighbour among tokens of positive weight).
* alpha, entropy and the TV loss within 1e-5 relative for float32 logits and
  2e-3 for bfloat16 logits (plus 1e-6 absolute, since entropy and alpha may
  be zero), gradients within 1e-4 absolute.
* flags must match exactly.
"""
from __future__ import annotations

import numpy as np

MARGIN = 1e-5
ERROR_BITS = 1 | 2 | 4 | 16 | 32  # every flag except ZERO_MASS (8)
GRAD_ATOL = 1e-4
ATOL = 1e-6


# Gumbel-max final draw: the device forms keys (ln w + G) in fp32 with
# approximate logarithms, and re-keys its two best candidates in double
# precision whenever they are near a tie; a draw counts as near its margin
# when the oracle's best and second best keys (natural-log units) are closer
# than this, the same 1e-5 as the other decisions.
GUMBEL_MARGIN = 1e-5


def gumbel_margins(orc: dict) -> dict:
    """An oracle gumbel_verify result in verify_report's terms: the final
    draw counts as near its margin when the top two keys are closer than
    GUMBEL_MARGIN."""
    o = dict(orc)
    o["cdf_margin"] = np.where(orc["gumbel_margin"] < GUMBEL_MARGIN, 0.0, 1.0)
    return o


def rtol_for(dtype: str) -> float:
    return 1e-5 if dtype == "f32" else 2e-3


def _relerr(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-30)


def _probs(z_row, T: float) -> np.ndarray:
    """float64 softmax(z / T) of one row; T = 0 is one-hot at the first arg max."""
    from . import softmax

    if T == 0.0:
        from . import _logits

        z, dt = _logits(np.asarray(z_row).reshape(1, -1))
        zf = z.astype(np.float64) if dt != 1 else (z.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        w = np.zeros(zf.shape[-1])
        w[int(np.argmax(zf[0]))] = 1.0
        return w
    return softmax(np.asarray(z_row).reshape(1, -1), T)[0]


def final_weights(x, b: int, n: int, mode: str = "rs", yhat=None) -> np.ndarray:
    """float64 weights of the final draw of sequence b after n accepted
    drafts ([BB] App. G.1; [EM] "Speculative Decoding"): at a rejection the
    residual max(0, p_n - q_n) (target-only: p_n with the proposed token
    removed), after gamma accepts p_gamma; a residual that sums to 0 falls
    back to p_n, as the library's ZERO_MASS rule does."""
    T = float(x.temperature[b])
    p = _probs(x.target[b, n], T)
    if n == x.gamma:
        return p
    if mode == "to":
        r = p.copy()
        r[int(yhat[b, n])] = 0.0
    else:
        r = np.maximum(p - _probs(x.draft[b, n], T), 0.0)
    return r if r.sum() > 0.0 else p


def final_weights_row(z_row, T: float) -> np.ndarray:
    """float64 weights of a draft-sampling draw: softmax(z / T) of the row
    (one-hot at the first arg max for T = 0) ([BB] App. G, G.1, G.2)."""
    return _probs(z_row, T)


def accept_ratio(x, b: int, i: int, mode: str = "rs", yhat=None) -> float:
    """p_i(y)/q_i(y) of the accept test of position i in float64 (target-only:
    p_i(yhat)); +inf when q(y) = 0 < p(y)."""
    T = float(x.temperature[b])
    p = _probs(x.target[b, i], T)
    if mode == "to":
        return float(p[int(yhat[b, i])])
    y = int(x.draft_ids[b, i])
    q = _probs(x.draft[b, i], T)
    if q[y] > 0.0:
        return float(p[y] / q[y])
    return np.inf if p[y] > 0.0 else np.nan


def cdf_token_ok(w: np.ndarray, v: int, u: float) -> bool:
    """Token v is a valid inverse-CDF draw of weights w at uniform u up to
    the margin: positive weight, and its CDF interval [C(v-1), C(v)] within
    MARGIN * R of u * R."""
    if not 0 <= v < w.shape[0] or not w[v] > 0.0:
        return False
    R = float(w.sum())
    c = np.cumsum(w)
    lo = float(c[v - 1]) if v > 0 else 0.0
    return lo - MARGIN * R <= u * R <= float(c[v]) + MARGIN * R


def gumbel_token_ok(w: np.ndarray, v: int, seed: int, offset: int, b: int, row: int) -> bool:
    """Token v is a valid Gumbel-max draw of weights w up to the margin:
    positive weight, and its key ln w_v + G_v within GUMBEL_MARGIN of the
    best key ([BB] App. G.2)."""
    from . import gumbel_noise

    if not 0 <= v < w.shape[0] or not w[v] > 0.0:
        return False
    G = gumbel_noise(seed, offset, b, row, 0, w.shape[0])
    with np.errstate(divide="ignore"):
        keys = np.where(w > 0.0, np.log(np.where(w > 0.0, w, 1.0)) + G, -np.inf)
    return bool(keys[v] >= keys.max() - GUMBEL_MARGIN)


def verify_report(tokens, accept_len, flags, orc: dict, draft_ids, gamma: int, V: int, dtype: str,
                  alpha=None, entropy=None, *, x=None, mode: str = "rs", seed: int = 0, offset: int = 0) -> dict:
    """Compare one verify call; returns a report dict (see assert_ok).

    A sequence whose tokens differ from the oracle's is accepted only when
    the difference is explained by a decision near its margin, and its
    output is checked for validity against float64 weights computed from
    the inputs `x` (target, draft, draft_ids, temperature, uniforms):
    * where the accept lengths differ, the first differing accept test is
      near its margin in the oracle, and every later test the GPU took
      agrees with the float64 test unless that one is near its margin;
    * the accepted prefix equals the draft tokens;
    * the drawn token has positive weight in the distribution it is drawn
      from (the residual max(0, p - q), p_gamma for the bonus, p without the
      proposed token for target-only acceptance), and it is the draw at the
      uniform up to the margin (inverse CDF: its CDF interval within
      MARGIN * R of u * R, i.e. the oracle's token or its neighbour among
      the tokens of positive weight; Gumbel-max: its key within
      GUMBEL_MARGIN of the best);
    * the padding after it is -1.
    rep["decisions"] counts the decisions the oracle took (accept tests and
    final draws); see near_margin_budget_ok.
    mode: "rs" (rejection sampling), "to" (target-only; draft_ids are the
    oracle's yhat) or "gumbel" (seed and offset of the noise)."""
    if x is None:
        raise ValueError("verify_report needs the inputs x to check near-margin outputs")
    B = accept_len.shape[0]
    rep = {"B": B, "exact": 0, "near_margin": 0, "decisions": 0, "mismatch": [], "flag_mismatch": [],
           "stats_bad": []}
    for b in range(B):
        if flags[b] != orc["flags"][b]:
            rep["flag_mismatch"].append((b, int(flags[b]), int(orc["flags"][b])))
            continue
        if orc["accept_len"][b] < 0:
            if accept_len[b] != -1 or np.any(tokens[b] != -1):
                rep["mismatch"].append((b, "flagged row outputs"))
            continue
        n_o = int(orc["accept_len"][b])
        rep["decisions"] += min(n_o + 1, gamma) + 1
        taken = orc["acc_margin"][b, : min(n_o + 1, gamma)]
        near = bool(np.any(taken < MARGIN)) or bool(orc["cdf_margin"][b] < MARGIN)
        same = accept_len[b] == n_o and np.array_equal(tokens[b], orc["tokens"][b])
        if same:
            rep["exact"] += 1
            continue
        if not near:
            rep["mismatch"].append((b, f"gpu n={int(accept_len[b])} tok={tokens[b].tolist()} "
                                       f"oracle n={n_o} tok={orc['tokens'][b].tolist()}"))
            continue
        rep["near_margin"] += 1
        why = _near_margin_invalid(tokens[b], int(accept_len[b]), n_o, orc, b, gamma, x, mode, draft_ids, seed,
                                   offset)
        if why:
            rep["mismatch"].append((b, "invalid near-margin output: " + why))
    if alpha is not None:
        rep.update(stats_report(alpha, entropy, orc, dtype, flags))
    return rep


def _near_margin_invalid(tok, n, n_o, orc, b, gamma, x, mode, draft_ids, seed, offset) -> str:
    """Why a near-margin sequence's output is not a valid one ('' if valid)."""
    if not 0 <= n <= gamma:
        return f"accept length {n}"
    if not np.array_equal(tok[:n], draft_ids[b, :n]):
        return "accepted prefix differs from the draft tokens"
    if np.any(tok[n + 1:] != -1):
        return "padding"
    if n != n_o:
        i = min(n, n_o)
        if not orc["acc_margin"][b, i] < MARGIN:
            return f"accept test {i} flipped away from its margin"
        # tests the oracle never took (the GPU accepted past the oracle's stop)
        for j in range(n_o + 1, min(n + 1, gamma)):
            ratio = accept_ratio(x, b, j, mode, draft_ids)
            u = float(x.uniforms[b, j])
            accept = u < ratio if np.isfinite(ratio) else bool(ratio > 0)
            if accept != (j < n) and not abs(u - ratio) < MARGIN:
                return f"accept test {j} disagrees with float64"
    w = final_weights(x, b, n, mode, draft_ids)
    v = int(tok[n])
    if mode == "gumbel":
        ok = gumbel_token_ok(w, v, seed, offset, b, n)
    else:
        ok = cdf_token_ok(w, v, float(x.uniforms[b, gamma]))
    if not ok:
        return f"drawn token {v} is not a valid draw (weight {w[v] if 0 <= v < w.shape[0] else 'n/a'})"
    return ""


def near_margin_budget_ok(rep: dict, frac: float = 0.01) -> bool:
    """Near-margin sequences stay below `frac` of the decisions taken."""
    return rep["near_margin"] <= frac * rep["decisions"]


def stats_report(alpha, entropy, orc: dict, dtype: str, flags=None) -> dict:
    rt = rtol_for(dtype)
    good = (orc["flags"] & ERROR_BITS) == 0  # rows without error bits
    ea = np.abs(alpha[good].astype(np.float64) - orc["alpha"][good])
    eh = np.abs(entropy[good].astype(np.float64) - orc["entropy"][good])
    bad_a = ea > rt * np.abs(orc["alpha"][good]) + ATOL
    bad_h = eh > rt * np.abs(orc["entropy"][good]) + ATOL
    out = {
        "alpha_max_abs": float(ea.max()) if ea.size else 0.0,
        "alpha_max_rel": float(_relerr(alpha[good], orc["alpha"][good]).max()) if ea.size else 0.0,
        "entropy_max_abs": float(eh.max()) if eh.size else 0.0,
        "entropy_max_rel": float(_relerr(entropy[good], orc["entropy"][good]).max()) if eh.size else 0.0,
        "stats_bad": [],
    }
    if bad_a.any():
        out["stats_bad"].append(("alpha", int(bad_a.sum())))
    if bad_h.any():
        out["stats_bad"].append(("entropy", int(bad_h.sum())))
    if not np.all(np.isnan(alpha[~good])) or not np.all(np.isnan(entropy[~good])):
        out["stats_bad"].append(("flagged rows not NaN", 1))
    if flags is not None and not np.array_equal(flags, orc["flags"]):
        out["stats_bad"].append(("flags", int((flags != orc["flags"]).sum())))
    return out


def diag_report(g: dict, orc: dict, dtype: str, logit_scale=None) -> dict:
    """Compare acceptance diagnostics.  Floats within the dtype's relative
    tolerance; the KL divergence is a difference of log-normalisers and
    weighted logit means, so its absolute tolerance also grows with the
    position's logit magnitude |z| / T (logit_scale [B, gamma]); yhat exact;
    rs_better exact except where the oracle's |d_TV - (1 - p(yhat))| is
    below MARGIN (counted as near-margin)."""
    rt = rtol_for(dtype)
    rep = {"B": int(orc["flags"].shape[0]), "near_margin": 0, "bad": []}
    if not np.array_equal(g["row_flags"], orc["flags"]):
        rep["bad"].append(("flags", int((g["row_flags"] != orc["flags"]).sum())))
    good = (orc["flags"] & ERROR_BITS) == 0
    for key in ("alpha", "ent_p", "ent_q", "p_yhat"):
        a = g[key][good].astype(np.float64)
        o = orc[key][good]
        e = np.abs(a - o)
        rep[key + "_max_abs"] = float(e.max()) if e.size else 0.0
        if np.any(~(e <= rt * np.abs(o) + ATOL)):
            rep["bad"].append((key, int((~(e <= rt * np.abs(o) + ATOL)).sum())))
    a = g["kl"][good].astype(np.float64)
    o = orc["kl"][good]
    fin = np.isfinite(o)
    if not np.array_equal(np.isfinite(a), fin) or np.any(a[~fin] != o[~fin]):
        rep["bad"].append(("kl infinities", int((np.isfinite(a) != fin).sum())))
    sc = np.zeros_like(o) if logit_scale is None else np.asarray(logit_scale, np.float64)[good]
    tol = rt * np.abs(o) + ATOL + 4e-7 * (1.0 + sc)
    e = np.where(fin, np.abs(np.where(fin, a, 0.0) - np.where(fin, o, 0.0)), 0.0)
    rep["kl_max_abs"] = float(e[fin].max()) if fin.any() else 0.0
    if np.any(~(e[fin] <= tol[fin])):
        rep["bad"].append(("kl", int((~(e[fin] <= tol[fin])).sum())))
    if not np.array_equal(g["yhat"][good], orc["yhat"][good]):
        rep["bad"].append(("yhat", int((g["yhat"][good] != orc["yhat"][good]).sum())))
    near = orc["boundary_margin"][good] < MARGIN
    rep["near_margin"] = int(near.sum())
    diff = (g["rs_better"][good] != orc["rs_better"][good]) & ~near
    if diff.any():
        rep["bad"].append(("rs_better", int(diff.sum())))
    bad_rows = ~good
    if bad_rows.any():
        for key in ("alpha", "ent_p", "ent_q", "kl", "p_yhat"):
            if not np.all(np.isnan(g[key][bad_rows])):
                rep["bad"].append((key + " of flagged rows not NaN", 1))
        for key in ("yhat", "rs_better"):
            if not np.all(g[key][bad_rows] == -1):
                rep["bad"].append((key + " of flagged rows not -1", 1))
    return rep


def tv_report(loss, alpha, grad, flags, orc: dict, dtype: str, target_f64=None, draft_f64=None,
              temperature: float = 1.0) -> dict:
    """Compare TV-loss outputs.  Rows (t, k) whose oracle log-ratio
    min_v |log q_v - log p_v| is below MARGIN sit on an indicator tie and are
    only checked for sum_j grad = 0; they are counted as near-margin."""
    rt = rtol_for(dtype)
    rep = {"positions": int(loss.shape[0]), "near_margin_rows": 0, "bad": []}
    if not np.array_equal(flags, orc["flags"]):
        rep["bad"].append(("flags", int((flags != orc["flags"]).sum())))
    good = orc["flags"] == 0
    el = np.abs(loss[good].astype(np.float64) - orc["loss"][good])
    ea = np.abs(alpha[good].astype(np.float64) - orc["alpha"][good])
    rep["loss_max_abs"] = float(el.max()) if el.size else 0.0
    rep["alpha_max_abs"] = float(ea.max()) if ea.size else 0.0
    if np.any(el > rt * np.abs(orc["loss"][good]) + ATOL):
        rep["bad"].append(("loss", int((el > rt * np.abs(orc["loss"][good]) + ATOL).sum())))
    if np.any(ea > rt * np.abs(orc["alpha"][good]) + ATOL):
        rep["bad"].append(("alpha", int((ea > rt * np.abs(orc["alpha"][good]) + ATOL).sum())))
    N, gamma = alpha.shape
    gmax = 0.0
    for t in range(N):
        if not good[t]:
            if np.any(grad[t] != 0):
                rep["bad"].append(("flagged grad not zero", t))
            continue
        for k in range(gamma):
            d = np.abs(grad[t, k].astype(np.float64) - orc["grad"][t, k])
            near = False
            if target_f64 is not None:
                lp = target_f64[t, k] / temperature
                lq = draft_f64[t, k] / temperature
                lp = lp - np.logaddexp.reduce(lp)
                lq = lq - np.logaddexp.reduce(lq)
                with np.errstate(invalid="ignore"):
                    gap = np.abs(lq - lp)
                near = bool(np.nanmin(gap) < MARGIN)
            if near and d.max() > GRAD_ATOL:
                rep["near_margin_rows"] += 1
                if abs(float(grad[t, k].astype(np.float64).sum())) > 1e-3:
                    rep["bad"].append(("near-margin row sum", (t, k)))
                continue
            gmax = max(gmax, float(d.max()))
            if d.max() > GRAD_ATOL:
                rep["bad"].append(("grad", (t, k, float(d.max()))))
    rep["grad_max_abs"] = gmax
    return rep


def assert_ok(rep: dict, what: str = "") -> None:
    problems = []
    for key in ("mismatch", "flag_mismatch", "stats_bad", "bad"):
        if rep.get(key):
            problems.append(f"{key}: {rep[key][:8]}")
    if problems:
        raise AssertionError(f"{what} parity failed: " + "; ".join(problems) + f" | report {_short(rep)}")


def _short(rep):
    return {k: v for k, v in rep.items() if not isinstance(v, list)}
