"""GPU parity of the CUDA path (through the C ABI) against the float64 oracle
on the same seeded inputs.  See oracle/compare.py for the bar."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import compare
from tests.gpu_util import ensure_library, kcode, tune, run_stats, run_tv, run_verify, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _check_verify(x, with_stats=False, what=""):
    g = run_verify(x, with_stats)
    o = oracle.verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms, want_stats=with_stats)
    rep = compare.verify_report(g["tokens"], g["accept_len"], g["row_flags"], o, x.draft_ids, x.gamma, x.V, x.dtype,
                                g["alpha"], g["entropy"], x=x)
    compare.assert_ok(rep, what)
    return rep, g, o


# ------------------------------------------------------------ verify -------

@pytest.mark.parametrize("with_stats", [False, True])
def test_verify_tiny_config(with_stats):
    x = W.config("tiny")
    rep, g, o = _check_verify(x, with_stats, "tiny")
    assert rep["exact"] + rep["near_margin"] == x.B


SWEEP = [
    # (V, dtype, gamma, T, forced cluster)
    (1, "f32", 3, 1.0, None),
    (7, "bf16", 3, 0.6, 4),
    (8, "bf16", 1, 1.7, None),
    (100, "f32", 7, 1.0, 16),
    (1000, "bf16", 3, 0.6, 2),
    (1024, "f32", 3, 1.7, 8),
    (4097, "bf16", 7, 1.0, 4),
    (4097, "f32", 1, 0.6, 16),
    (40000, "bf16", 3, 1.0, 8),
    (40003, "f32", 3, 0.8, 16),
]


@pytest.mark.parametrize("V,dtype,gamma,T,C", SWEEP)
@pytest.mark.parametrize("with_stats", [False, True])
def test_verify_sweep(V, dtype, gamma, T, C, with_stats):
    x = W.verify_inputs(f"sweep{V}", 24, gamma, V, dtype, 1000 + V + gamma, family="sigma",
                        sigmas=np.linspace(0.5, 4.0, 24), delta=np.linspace(0.0, 1.0, 24), temperature=T)
    with tune(cluster_size=C):
        rep, g, o = _check_verify(x, with_stats, f"sweep V={V} {dtype} gamma={gamma} C={C}")
    assert compare.near_margin_budget_ok(rep), rep


@pytest.mark.parametrize("V,dtype,gamma,T,C", [s for s in SWEEP if s[0] % (4 if s[1] == "f32" else 8) == 0])
def test_verify_sweep_resident_kernel(V, dtype, gamma, T, C):
    """Aligned rows without statistics normally take the streaming kernel;
    the cluster-resident kernel must agree as well."""
    x = W.verify_inputs(f"sweep{V}", 24, gamma, V, dtype, 1000 + V + gamma, family="sigma",
                        sigmas=np.linspace(0.5, 4.0, 24), delta=np.linspace(0.0, 1.0, 24), temperature=T)
    with tune(cluster_size=C, verify_kernel=kcode("resident")):
        rep, g, o = _check_verify(x, False, f"resident V={V} {dtype} gamma={gamma} C={C}")
    assert compare.near_margin_budget_ok(rep), rep


@pytest.mark.parametrize("ring,depth,C,clusters,chunk", [(2, 0, 4, None, None), (2, 1, 8, 3, None),
                                                         (3, 5, None, None, None), (8, 5, 2, 5, 128),
                                                         (4, 0, 16, 2, None), (3, 2, 1, 7, 192), (2, 3, 4, 1, 192),
                                                         (2, 5, 1, 3, 192), (2, 5, 2, None, 128)])
def test_verify_stream_ring_variants(ring, depth, C, clusters, chunk):
    """Ring slots, look-ahead depth, cluster size, chunk size and several
    sequences per cluster (capped grid) on rows with many rejections."""
    B = 40
    x = W.verify_inputs("ring", B, 5, 40000, "bf16", 77, family="sigma", sigmas=np.linspace(0.5, 6.0, B),
                        delta=np.linspace(0.0, 2.0, B), temperature=np.linspace(0.6, 1.3, B))
    with tune(ring_slots=ring, lookahead=depth + 1, cluster_size=C, max_clusters=clusters,
             chunk_vectors=chunk):
        rep, g, o = _check_verify(x, False, f"ring={ring} depth={depth} C={C} clusters={clusters} chunk={chunk}")
    n = g["accept_len"]
    assert (n == x.gamma).any() and (n < x.gamma).any() and (n == 0).any()


def test_verify_stream_bad_rows_between_good_ones():
    """Flagged sequences in the middle of a cluster's list: the look-ahead
    into them is dropped and the following sequences stay exact."""
    B = 64
    x = W.verify_inputs("mix", B, 3, 8192, "f32", 78, family="sigma", sigmas=np.linspace(1.0, 5.0, B),
                        delta=np.linspace(0.1, 1.5, B))
    x.temperature[5::9] = -1.0
    x.draft_ids[7::11, 1] = -4
    x.uniforms[3::13, 3] = 1.5
    x.target[10::17, 1, 100] = np.inf
    with tune(cluster_size=2, max_clusters=5):
        rep, g, o = _check_verify(x, False, "bad rows mixed")
    np.testing.assert_array_equal(g["row_flags"], o["flags"])
    assert (o["flags"] != 0).sum() >= 10


@pytest.mark.parametrize("gamma", [8, 9, 31, 32])
def test_verify_long_draft(gamma):
    """gamma = 8 is the streaming kernel's limit; longer drafts take the
    cluster-resident kernel."""
    x = W.verify_inputs("long", 6, gamma, 2048, "bf16", 79, family="sigma", sigmas=1.0, delta=0.0)
    j = min(20, gamma - 2)
    x.draft[2, j] = x.draft[2, j] ^ np.uint16(0x0040)  # a perturbed row late in one sequence
    rep, g, o = _check_verify(x, False, f"gamma={gamma}")
    assert rep["exact"] + rep["near_margin"] == x.B


def _random_configs(n, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = "bf16" if rng.random() < 0.6 else "f32"
        V = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 5000)), int(rng.integers(5000, 70000))]))
        out.append((i, dtype, V, int(rng.integers(1, 21)), int(rng.integers(1, 9))))
    return out


@pytest.mark.parametrize("i,dtype,V,B,gamma", _random_configs(24))
def test_randomized_shapes(i, dtype, V, B, gamma):
    """Seeded random shapes (V from 1 to 70,000, odd sizes that leave rows
    unaligned included; B up to 20; gamma up to 8; per-sequence temperatures
    with greedy rows; logit scales and draft offsets spread wide): verify
    without and with statistics (a greedy row with statistics is flagged, as
    documented) and row statistics against the oracle, and draft sampling by
    both draws where the rows are whole 16-byte vectors."""
    rng = np.random.default_rng(9000 + i)
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    T[rng.random(B) < 0.15] = 0.0
    x = W.verify_inputs(f"rand{i}", B, gamma, V, dtype, 9100 + i, family="sigma",
                        sigmas=rng.uniform(0.2, 12.0, B), delta=rng.uniform(0.0, 1.5, B), temperature=T)
    what = f"random {i}: {dtype} V={V} B={B} gamma={gamma}"
    rep, g, o = _check_verify(x, False, what)  # T = 0 rows are greedy sequences
    assert rep["exact"] + rep["near_margin"] == x.B
    rep, g, o = _check_verify(x, True, what + " with stats")  # greedy rows with statistics are flagged
    assert rep["exact"] + rep["near_margin"] + int((o["accept_len"] < 0).sum()) == x.B
    gs = run_stats(x)
    os_ = oracle.row_stats(x.target, x.draft, x.temperature)
    compare.assert_ok(compare.stats_report(gs["alpha"], gs["entropy"], os_, dtype, gs["row_flags"]), f"random {i} stats")
    if V % (16 // (2 if dtype == "bf16" else 4)) == 0:
        z = x.draft.reshape(B * gamma, V)
        Tz = np.repeat(x.temperature, gamma).astype(np.float32)
        u = x.uniforms[:, :gamma].reshape(-1).copy()
        for method in ("multinomial", "gumbel"):
            _check_draft(z, Tz, u, method, 40 + i, i, dtype, f"random {i} draft {method}")


def test_verify_plan_kernels():
    import mtp_speculative_decoding_row_gb300 as mtp
    p = mtp.mtp_query_plan("verify", "bf16", 64, 3, 151936)
    assert p["resident_drafts"] > 0  # streaming kernel: ring slots per warp
    q = mtp.mtp_query_plan("verify_resident", "bf16", 64, 3, 151936)
    assert q["resident_drafts"] == 0
    with tune(verify_kernel=kcode("resident")):
        assert mtp.mtp_query_plan("verify", "bf16", 64, 3, 151936)["resident_drafts"] == 0


def test_draft_sample_plans():
    """Both draft-sampling plans count rows as units: at most one cluster per
    row.  Inverse CDF runs on the streaming kernel (ring slots per warp); the
    Gumbel-max plan is the one-pass kernel's (no ring, clusters of at most 8)."""
    import mtp_speculative_decoding_row_gb300 as mtp
    for op in ("draft_sample", "draft_sample_gumbel"):
        p = mtp.mtp_query_plan(op, "bf16", 192, 3, 151936)
        assert 1 <= p["clusters"] <= 192 and p["cluster_size"] >= 1 and p["smem_bytes"] > 0, (op, p)
    assert mtp.mtp_query_plan("draft_sample", "bf16", 192, 3, 151936)["resident_drafts"] >= 2
    g = mtp.mtp_query_plan("draft_sample_gumbel", "bf16", 192, 3, 151936)
    assert g["resident_drafts"] == 0 and g["cluster_size"] <= 8, g
    small = mtp.mtp_query_plan("draft_sample_gumbel", "bf16", 3, 3, 151936)
    assert small["clusters"] <= 3


@pytest.mark.parametrize("name,kernel", [("verify64", None), ("rl512", None), ("deep256", None),
                                         ("verify64", "resident"), ("rl512", "resident")])
def test_verify_full_configs(name, kernel):
    x = W.config(name)
    with tune(verify_kernel=kcode(kernel)):
        rep, g, o = _check_verify(x, x.want_stats, name)
    assert rep["exact"] + rep["near_margin"] == x.B
    assert compare.near_margin_budget_ok(rep), rep  # near-margin sequences below 1 % of the decisions
    # both the accept path and the residual path occur at these sizes
    n = g["accept_len"]
    assert (n == x.gamma).any() and (n < x.gamma).any()
    print(name, {k: v for k, v in rep.items() if not isinstance(v, list)})


def test_verify_equal_rows_accept_all():
    """delta = 0 rows give q == p: every draft accepted, alpha = 1."""
    x = W.verify_inputs("eq", 16, 5, 5000, "bf16", 7, family="sigma", sigmas=3.0, delta=0.0)
    g = run_verify(x, with_stats=True)
    assert np.all(g["accept_len"] == 5)
    np.testing.assert_array_equal(g["tokens"][:, :5], x.draft_ids)
    np.testing.assert_allclose(g["alpha"], 1.0, atol=2e-6)


def _zero_mass_inputs(B=8, V=1024):
    """Verify inputs (gamma = 1, fp32) whose every sequence rejects its draft
    token y with a residual max(0, p - q) that is exactly zero: the draft row
    equals the target row except at y, where the logits are -300 (target) and
    -299 (draft).  At T = 1 that index's weight underflows next to the others
    in single and in double precision, so both normalisers, and with them p
    and q away from y, agree bit for bit; at y itself q > p, and u = 0.9
    rejects (u q(y) >= p(y)).  The rounding case the pages' two-pass CDF
    leaves open: the draw falls back to p and the row is flagged ZERO_MASS."""
    rng = np.random.default_rng(4321)
    g = 1
    t = (rng.standard_normal((B, g + 1, V)) * 2.0).astype(np.float32)
    y = rng.integers(0, V, size=(B, g)).astype(np.int32)
    d = t[:, :g].copy()
    for b in range(B):
        t[b, 0, y[b, 0]] = -300.0
        d[b, 0, y[b, 0]] = -299.0
    u = np.full((B, g + 1), 0.9, np.float32)
    u[:, g] = rng.random(B).astype(np.float32)
    return W.VerifyInputs("zeromass", B, g, V, "f32", t, d, y, np.ones(B, np.float32), u)


@pytest.mark.parametrize("kernel", ["stream", "resident", "stats", "gumbel"])
def test_zero_mass_residual_fallback(kernel):
    """A rejection whose residual mass is exactly zero (see
    _zero_mass_inputs): every kernel path that takes the residual draw (the
    streaming and the cluster-resident verify, verify with statistics, the
    Gumbel-max draw) rejects, flags MTP_ROW_ZERO_MASS, draws from p instead,
    and matches the oracle, which takes the same fallback."""
    import mtp_speculative_decoding_row_gb300 as mtp
    x = _zero_mass_inputs()
    if kernel == "gumbel":
        _, g, o = _check_gumbel(x, 77, 3, "zero-mass gumbel")
    else:
        with tune(verify_kernel=kcode("resident") if kernel == "resident" else 0):
            _, g, o = _check_verify(x, with_stats=kernel == "stats", what=f"zero-mass {kernel}")
    assert np.all(o["flags"] == mtp.ROW_ZERO_MASS) and np.all(g["row_flags"] == mtp.ROW_ZERO_MASS)
    assert np.all(g["accept_len"] == 0)
    assert np.all((g["tokens"][:, 0] >= 0) & (g["tokens"][:, 0] != x.draft_ids[:, 0]))


def test_verify_deterministic():
    x = W.verify_inputs("det", 32, 3, 30000, "bf16", 8, family="sigma", sigmas=np.linspace(1, 6, 32), delta=0.4)
    a = run_verify(x, True)
    b = run_verify(x, True)
    for k in ("tokens", "accept_len", "alpha", "entropy", "row_flags"):
        np.testing.assert_array_equal(a[k], b[k])


def test_verify_output_law_chi_square():
    """Output-token law equals p ("RS preserves the exact target
    distribution"): one V = 8 row pair replicated 2^20 times with fresh
    uniforms and draft ids ~ q; chi-square at a fixed seed."""
    B, V = 1 << 20, 8
    rng = np.random.Generator(np.random.Philox(4242))
    zt = rng.standard_normal((2, V)).astype(np.float32) * 1.3
    zd = (zt[:1] + rng.standard_normal((1, V)).astype(np.float32) * 0.9).astype(np.float32)
    q = np.exp(zd[0].astype(np.float64) - zd[0].max())
    q /= q.sum()
    ids = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
    u = rng.random((B, 2), dtype=np.float32)
    t = torch.from_numpy(np.broadcast_to(zt, (B, 2, V)).copy()).cuda()
    d = torch.from_numpy(np.broadcast_to(zd, (B, 1, V)).copy()).cuda()
    import mtp_speculative_decoding_row_gb300 as mtp
    out = mtp.mtp_rs_verify(t, d, torch.from_numpy(ids).cuda(), torch.ones(B, device="cuda"),
                            torch.from_numpy(u).cuda())
    first = out.tokens[:, 0].cpu().numpy()
    p = oracle.softmax(zt[0])
    counts = np.bincount(first, minlength=V)
    chi2 = ((counts - B * p) ** 2 / (B * p)).sum()
    assert chi2 < 24.3, (chi2, counts, B * p)  # 0.999 quantile, 7 dof


# --------------------------------------------- greedy and target-only ------

def _check_to_verify(x, what=""):
    import mtp_speculative_decoding_row_gb300 as mtp
    out = mtp.mtp_to_verify(to_dev(x.target), to_dev(x.draft), to_dev(x.temperature), to_dev(x.uniforms))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out._asdict().items()}
    o = oracle.to_verify(x.target, x.draft, x.temperature, x.uniforms)
    rep = compare.verify_report(g["tokens"], g["accept_len"], g["row_flags"], o, o["yhat"], x.gamma, x.V, x.dtype,
                                x=x, mode="to")
    compare.assert_ok(rep, what)
    exact = (g["accept_len"] == o["accept_len"]) & np.all(g["tokens"] == o["tokens"], axis=1)
    np.testing.assert_array_equal(g["draft_tokens"][exact], o["yhat"][exact])
    return rep, g, o


TO_SWEEP = [
    # (V, dtype, gamma, C, clusters)
    (1024, "f32", 3, None, None),
    (4096, "bf16", 5, 4, None),
    (40000, "bf16", 3, 8, None),
    (40000, "f32", 8, 16, None),
    (40000, "f32", 8, 4, 2),
    (151936, "bf16", 3, None, None),
]


@pytest.mark.parametrize("V,dtype,gamma,C,clusters", TO_SWEEP)
def test_to_verify(V, dtype, gamma, C, clusters):
    """Target-only verification: arg max drafts, u < p(y), residual p without
    y; a quarter of the rows greedy (T = 0), mixed with sampled rows on the
    same cluster."""
    B = 32
    x = W.verify_inputs(f"to{V}", B, gamma, V, dtype, 3000 + V + gamma, family="sigma",
                        sigmas=np.linspace(0.5, 6.0, B), delta=np.linspace(0.0, 1.5, B),
                        temperature=np.where(np.arange(B) % 4 == 3, 0.0, np.linspace(0.6, 1.3, B)))
    with tune(cluster_size=C, max_clusters=clusters):
        rep, g, o = _check_to_verify(x, f"to V={V} {dtype} gamma={gamma} C={C} clusters={clusters}")
    n = g["accept_len"]
    assert (n > 0).any() and (n < gamma).any()


def test_to_verify_full_config():
    x = W.config("verify64")
    rep, g, o = _check_to_verify(x, "to verify64")
    assert rep["exact"] + rep["near_margin"] == x.B and compare.near_margin_budget_ok(rep), rep


@pytest.mark.parametrize("V,dtype,gamma,kernel,clusters", [(30000, "bf16", 3, None, None),
                                                           (4096, "f32", 5, "resident", None),
                                                           (4097, "bf16", 3, None, None),
                                                           (2048, "bf16", 12, None, None),
                                                           (40000, "f32", 8, None, 2),
                                                           (30000, "bf16", 5, "resident", 3)])
def test_greedy_rs_verify(V, dtype, gamma, kernel, clusters):
    """T = 0 rows of mtp_rs_verify are greedy: accept while the draft is the
    target's arg max (streaming kernel, cluster-resident kernel, unaligned
    rows, gamma > 8, and greedy stops followed by more sequences on the same
    cluster, whose look-ahead rows must be dropped)."""
    B = 24
    x = W.verify_inputs(f"greedy{V}", B, gamma, V, dtype, 3100 + V, family="sigma", sigmas=np.linspace(1, 5, B),
                        delta=np.linspace(0.0, 0.8, B), temperature=np.where(np.arange(B) % 2 == 0, 0.0, 1.0))
    # half of the greedy rows draft the target's arg max at every position
    tgt = W.bf16_bits_to_f32(x.target) if dtype == "bf16" else x.target
    am = tgt[:, :gamma].argmax(-1).astype(np.int32)
    x.draft_ids[::4] = am[::4]
    with tune(verify_kernel=kcode(kernel), max_clusters=clusters):
        rep, g, o = _check_verify(x, False, f"greedy V={V} gamma={gamma} kernel={kernel} clusters={clusters}")
    greedy = x.temperature == 0
    assert np.all(g["accept_len"][::4] == gamma)
    assert rep["exact"] == B
    np.testing.assert_array_equal(g["tokens"][greedy], o["tokens"][greedy])


# ------------------------------------------------------------- stats -------

@pytest.mark.parametrize("V,dtype,gamma,C,kernel", [(1024, "f32", 3, None, None), (4097, "bf16", 5, 8, None),
                                                    (151936, "bf16", 3, None, None), (30001, "f32", 2, 16, None),
                                                    (40000, "bf16", 10, None, None),
                                                    (1024, "f32", 3, None, "stream"), (40000, "f32", 7, 4, "stream"),
                                                    (40000, "bf16", 8, 16, "stream"), (64, "f32", 3, 16, "stream"),
                                                    (151936, "bf16", 3, None, "stream"),
                                                    (4097, "bf16", 5, 8, "stream"),
                                                    (1024, "f32", 3, None, "resident"),
                                                    (151936, "bf16", 3, None, "resident"),
                                                    (1024, "f32", 3, 2, "tmem"), (151936, "f32", 7, 8, "tmem"),
                                                    (40000, "bf16", 8, 4, "tmem"), (64, "f32", 3, 8, "tmem"),
                                                    (151936, "bf16", 1, None, "tmem")])
def test_row_stats(V, dtype, gamma, C, kernel):
    """Row statistics on the planner's kernel (cluster-resident), and on the
    streaming row-pair and TMEM-resident kernels when asked for (V = 64 over
    64 or 128 segments leaves most warps without vocabulary)."""
    x = W.verify_inputs("stats", 12, gamma, V, dtype, 2000 + V, family="sigma", sigmas=np.linspace(0.3, 9, 12),
                        delta=np.linspace(0, 1.5, 12), temperature=np.linspace(0.6, 1.4, 12))
    with tune(cluster_size=C, stats_kernel=kcode(kernel)):
        g = run_stats(x)
    o = oracle.row_stats(x.target, x.draft, x.temperature)
    rep = compare.stats_report(g["alpha"], g["entropy"], o, dtype, g["row_flags"])
    compare.assert_ok(rep, f"stats V={V}")


@pytest.mark.parametrize("clusters,C", [(1, None), (3, 8), (2, 4)])
def test_row_stats_tmem_sequences_and_flags(clusters, C):
    """The TMEM-resident statistics kernel with several sequences per
    cluster (the exchange barriers reused sequence after sequence), bad
    temperatures (T = 0 included) skipped between good sequences, and NaN
    and +inf logits flagged."""
    B, gamma, V = 11, 4, 40000
    x = W.verify_inputs("stm", B, gamma, V, "f32", 2150 + clusters, family="sigma", sigmas=np.linspace(0.5, 7, B),
                        delta=np.linspace(0, 1.2, B), temperature=np.linspace(0.6, 1.4, B))
    x.temperature[[2, 7]] = [0.0, -1.0]
    x.target[4, 1, 123] = np.nan
    x.draft[9, 3, 39999] = np.inf
    with tune(stats_kernel=kcode("tmem"), max_clusters=clusters, cluster_size=C):
        g = run_stats(x)
    o = oracle.row_stats(x.target, x.draft, x.temperature)
    np.testing.assert_array_equal(g["row_flags"], o["flags"])
    assert list(np.nonzero(o["flags"])[0]) == [2, 4, 7, 9]
    rep = compare.stats_report(g["alpha"], g["entropy"], o, "f32", g["row_flags"])
    compare.assert_ok(rep, f"tmem stats clusters={clusters}")


def test_row_stats_deep_config():
    x = W.config("deep256")
    g = run_stats(x)
    o = oracle.row_stats(x.target, x.draft, x.temperature)
    rep = compare.stats_report(g["alpha"], g["entropy"], o, x.dtype, g["row_flags"])
    compare.assert_ok(rep, "deep256 stats")
    # alpha = 1 - TV against the oracle's independent TV
    np.testing.assert_allclose(g["alpha"], 1 - o["tv"], rtol=0, atol=1e-5)


# ------------------------------------------------- Gumbel-max final draw ---

def _check_gumbel(x, seed, offset, what=""):
    import mtp_speculative_decoding_row_gb300 as mtp
    out = mtp.mtp_gumbel_verify(to_dev(x.target), to_dev(x.draft), to_dev(x.draft_ids), to_dev(x.temperature),
                                to_dev(x.uniforms), seed, offset)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out._asdict().items() if v is not None}
    o = oracle.gumbel_verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms, seed, offset)
    rep = compare.verify_report(g["tokens"], g["accept_len"], g["row_flags"], compare.gumbel_margins(o), x.draft_ids,
                                x.gamma, x.V, x.dtype, x=x, mode="gumbel", seed=seed, offset=offset)
    compare.assert_ok(rep, what)
    return rep, g, o


GB_SWEEP = [
    # (V, dtype, gamma, C)
    (1024, "f32", 3, None),
    (4096, "bf16", 5, 4),
    (40000, "f32", 8, 16),
    (40000, "bf16", 3, 2),
    (30000, "f32", 4, 1),
    (151936, "bf16", 3, None),
]


@pytest.mark.parametrize("V,dtype,gamma,C", GB_SWEEP)
def test_gumbel_verify(V, dtype, gamma, C):
    """Rejection sampling with the Gumbel-max final draw (Philox noise in the
    kernel) against the oracle: residual and bonus draws, greedy rows
    (T = 0), a bad draft id; u[:, gamma] is not read."""
    B = 32
    x = W.verify_inputs(f"gb{V}", B, gamma, V, dtype, 5000 + V + gamma, family="sigma",
                        sigmas=np.linspace(0.5, 6.0, B), delta=np.linspace(0.0, 1.2, B),
                        temperature=np.where(np.arange(B) % 8 == 7, 0.0, np.linspace(0.6, 1.3, B)))
    x.uniforms[:, gamma] = 3.0  # not a valid uniform: must be ignored
    x.draft_ids[9, 0] = V + 5
    seed, offset = (1 << 40) + 12345, 7
    with tune(cluster_size=C):
        rep, g, o = _check_gumbel(x, seed, offset, f"gumbel V={V} {dtype} gamma={gamma} C={C}")
        assert g["row_flags"][9] == 2 and (g["row_flags"][np.arange(B) != 9] & 31 == 0).all()
        n = g["accept_len"]
        assert (n == gamma).any() and (n < gamma).any()
        # same stream: same tokens; another offset: other final tokens
        _, g2, _ = _check_gumbel(x, seed, offset, "repeat")
        np.testing.assert_array_equal(g["tokens"], g2["tokens"])
        _, g3, _ = _check_gumbel(x, seed, offset + 1, "offset + 1")
    sampled = (x.temperature > 0) & (g["row_flags"] == 0)
    fin = lambda t, a: t[np.arange(B), np.maximum(a, 0)]  # noqa: E731
    assert (fin(g["tokens"], n)[sampled] != fin(g3["tokens"], g3["accept_len"])[sampled]).any()


def test_gumbel_verify_full_config():
    x = W.config("verify64")
    rep, g, o = _check_gumbel(x, 2024, 0, "gumbel verify64")
    assert rep["exact"] + rep["near_margin"] == x.B and compare.near_margin_budget_ok(rep), rep


def test_streaming_modes_f32_full_vocab():
    """float32 rows at V = 151,936 through the three verify modes of the
    streaming kernel (rejection sampling, target-only, Gumbel-max), with a
    spread of entropies and temperatures."""
    B = 12
    x = W.verify_inputs("f32full", B, 3, W.V_QWEN, "f32", 4242, family="sigma", sigmas=np.linspace(0.5, 6.0, B),
                        delta=0.5, temperature=np.linspace(0.6, 1.4, B))
    assert compare_plan_streams("verify", x) and compare_plan_streams("to_verify", x)
    rep, g, o = _check_verify(x, False, "f32 full vocab")
    assert rep["exact"] + rep["near_margin"] == B
    rep, g, o = _check_to_verify(x, "f32 full vocab, target-only")
    assert rep["exact"] + rep["near_margin"] == B
    rep, g, o = _check_gumbel(x, 77, 3, "f32 full vocab, Gumbel-max")
    assert rep["exact"] + rep["near_margin"] == B


def compare_plan_streams(op, x):
    """True when the call would take the streaming kernel (ring slots > 0)."""
    import mtp_speculative_decoding_row_gb300 as mtp
    return mtp.mtp_query_plan(op, x.dtype, x.B, x.gamma, x.V)["resident_drafts"] > 0


def test_verify_in_cuda_graph():
    """mtp_rs_verify captured once in a CUDA graph on a side stream and
    replayed on two input sets copied into the captured buffers: the same
    results as the oracle for each set (no per-call host state is baked into
    the launch)."""
    import mtp_speculative_decoding_row_gb300 as mtp
    xs = [W.verify_inputs(f"graph{i}", 16, 3, 40000, "bf16", 5150 + i, family="sigma",
                          sigmas=np.linspace(1.0, 5.0, 16), delta=0.4) for i in range(2)]
    bufs = [to_dev(a) for a in (xs[0].target, xs[0].draft, xs[0].draft_ids, xs[0].temperature, xs[0].uniforms)]
    out = mtp.mtp_rs_verify(*bufs)  # plan caches and outputs before capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            mtp.mtp_rs_verify(*bufs, out=out, stream=s)
    torch.cuda.synchronize()
    for x in reversed(xs):
        for dst, src in zip(bufs, (x.target, x.draft, x.draft_ids, x.temperature, x.uniforms)):
            dst.copy_(to_dev(src))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        g = {k: (v.cpu().numpy() if v is not None else None) for k, v in out._asdict().items()}
        o = oracle.verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms, want_stats=False)
        rep = compare.verify_report(g["tokens"], g["accept_len"], g["row_flags"], o, x.draft_ids, x.gamma, x.V,
                                    x.dtype, x=x)
        compare.assert_ok(rep, "graph replay")
        assert rep["exact"] + rep["near_margin"] == x.B


# ------------------------------------------------------- draft sampling ----

def _draft_rows(V, dtype, gamma, seed, B=16):
    x = W.verify_inputs(f"ds{V}", B, gamma, V, dtype, seed, family="sigma", sigmas=np.linspace(0.4, 7.0, B),
                        delta=0.4, temperature=np.linspace(0.6, 1.3, B))
    z = x.draft.reshape(B * gamma, V)
    T = np.repeat(x.temperature, gamma).astype(np.float32)
    T[5::11] = 0.0  # greedy rows
    u = x.uniforms[:, :gamma].reshape(-1).copy()
    return z, T, u


def _check_draft(z, T, u, method, seed, offset, dtype, what):
    import mtp_speculative_decoding_row_gb300 as mtp
    out = mtp.mtp_draft_sample(to_dev(z), to_dev(T), to_dev(u), method=method, seed=seed, offset=offset)
    torch.cuda.synchronize()
    ids, flags = out.ids.cpu().numpy(), out.row_flags.cpu().numpy()
    o = oracle.draft_sample(z, T, u, method=method, seed=seed, offset=offset)
    np.testing.assert_array_equal(flags, o["flags"], err_msg=what)
    lim = compare.GUMBEL_MARGIN if method == "gumbel" else compare.MARGIN
    near = o["margin"] < lim
    bad = (ids != o["ids"]) & ~near
    assert not bad.any(), (what, np.nonzero(bad)[0][:8], ids[bad][:8], o["ids"][bad][:8])
    # a draw within rounding of a CDF breakpoint may take the neighbouring
    # index (flat rows at large V put many draws there); a near-tie of two
    # Gumbel keys may take the other key's index
    moved = (ids != o["ids"]) & near
    assert np.all((ids[moved] >= 0) & (ids[moved] < z.shape[1])), what
    if method == "multinomial":
        assert np.all(np.abs(ids[moved] - o["ids"][moved]) == 1), (what, ids[moved], o["ids"][moved])
    for r in np.nonzero(moved)[0]:  # positive weight, and the draw at its uniform or noise up to the margin
        w = compare.final_weights_row(z[r], float(T[r]))
        ok = (compare.gumbel_token_ok(w, int(ids[r]), seed, offset, int(r), 0) if method == "gumbel"
              else compare.cdf_token_ok(w, int(ids[r]), float(u[r])))
        assert ok, (what, int(r), int(ids[r]), int(o["ids"][r]))
    return ids, o


@pytest.mark.parametrize("method", ["multinomial", "gumbel"])
@pytest.mark.parametrize("V,dtype,C", [(1024, "f32", None), (4096, "bf16", 4), (40000, "f32", 16),
                                       (30000, "bf16", 1), (151936, "bf16", None)])
def test_draft_sample(V, dtype, C, method):
    """One draft token per row from softmax(z / T): inverse CDF with the
    caller's uniforms, or Gumbel-max with in-kernel Philox noise; T = 0
    rows are greedy."""
    z, T, u = _draft_rows(V, dtype, 3, 6000 + V)
    with tune(cluster_size=C):
        ids, o = _check_draft(z, T, u, method, 99, 4, dtype, f"draft sample V={V} {dtype} C={C} {method}")
    assert len(np.unique(ids)) > len(ids) // 4  # rows differ: the draws are not all one token


@pytest.mark.parametrize("C,clusters", [(1, 7), (2, 5), (8, 3), (None, None)])
def test_draft_sample_gumbel_rows_per_cluster(C, clusters):
    """The one-pass Gumbel-max kernel with several rows per persistent
    cluster (its records alternate between two buffers by row), across
    cluster sizes 1-8, with greedy rows, a NaN row and a bad temperature in
    between: draws and flags against the oracle."""
    z, T, u = _draft_rows(3000, "bf16", 3, 777, B=30)
    z = z.copy()
    z[17, 123] = 0x7FC0  # NaN (bf16 bits)
    T[40] = -1.0
    with tune(cluster_size=C, max_clusters=clusters):
        ids, o = _check_draft(z, T, u, "gumbel", 5, 2, "bf16", f"gumbel rows per cluster C={C} clusters={clusters}")
    assert o["flags"][17] != 0 and o["flags"][40] != 0
    assert np.count_nonzero(ids >= 0) >= len(ids) - 2


def _near_tie_rows(R, V, seed, offset, lo=1.5e-5, hi=5e-4, row=0):
    """Rows whose two largest logits are equal (5.0, exact in bf16 too), at
    the two indices whose Gumbel noise (the draws' counter-based noise of
    sequence r, row `row`) is closest within [lo, hi): their keys ln w + G
    differ by that gap, far above every other key (the rest is -30)."""
    z = np.full((R, V), -30.0, np.float32)
    gaps = np.empty(R)
    for r in range(R):
        G = oracle.gumbel_noise(seed, offset, r, row, 0, V)
        order = np.argsort(G)
        d = np.diff(G[order])
        ok = np.nonzero((d >= lo) & (d < hi))[0]
        i = ok[np.argmin(d[ok])] if r % 2 == 0 else ok[-1]
        z[r, order[i]] = z[r, order[i + 1]] = 5.0
        gaps[r] = d[i]
    return z, gaps


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gumbel_near_ties_resolved(dtype):
    """Two candidates whose Gumbel keys differ by 1.5e-5 to 5e-4 (natural-log
    units): the fp32 keys cannot order them reliably, the kernel's
    double-precision re-keying of its two best candidates must, so the
    draws equal the oracle's exactly (every gap is above GUMBEL_MARGIN)."""
    import mtp_speculative_decoding_row_gb300 as mtp
    R, V, seed, offset = 48, 512, 31337, 5
    z, gaps = _near_tie_rows(R, V, seed, offset)
    zs = W.to_bf16_bits(z) if dtype == "bf16" else z
    o = oracle.draft_sample(zs, np.ones(R, np.float32), None, method="gumbel", seed=seed, offset=offset)
    assert (o["margin"] >= compare.GUMBEL_MARGIN).all() and (o["margin"] < 1e-3).all()
    np.testing.assert_allclose(o["margin"], gaps, rtol=1e-6)
    out = mtp.mtp_draft_sample(to_dev(zs), torch.ones(R, device="cuda"), None, method="gumbel", seed=seed,
                               offset=offset)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.ids.cpu().numpy(), o["ids"])


def test_gumbel_verify_bonus_near_ties_resolved():
    """The same near-ties as the bonus draw of Gumbel-max verification: every
    draft accepted (draft row = target row 0), row gamma = 1 holds the tie."""
    import mtp_speculative_decoding_row_gb300 as mtp
    B, V, seed, offset = 32, 512, 4242, 9
    z1, gaps = _near_tie_rows(B, V, seed, offset, row=1)
    rng = np.random.default_rng(5)
    t = np.stack([rng.standard_normal((B, V)).astype(np.float32), z1], axis=1)
    d = t[:, :1].copy()
    ids = rng.integers(0, V, (B, 1)).astype(np.int32)
    T = np.ones(B, np.float32)
    u = rng.random((B, 2), dtype=np.float32)
    o = oracle.gumbel_verify(t, d, ids, T, u, seed, offset)
    assert (o["accept_len"] == 1).all() and (o["gumbel_margin"] >= compare.GUMBEL_MARGIN).all()
    out = mtp.mtp_gumbel_verify(to_dev(t), to_dev(d), to_dev(ids), to_dev(T), to_dev(u), seed, offset)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.tokens.cpu().numpy(), o["tokens"])


def test_draft_sample_bad_rows_and_full_size():
    """Bad temperature / uniform / NaN rows in between good ones, and the
    verify64 draft rows (192 rows of V = 151,936 bf16) against the oracle."""
    z, T, u = _draft_rows(8192, "f32", 2, 6100, B=20)
    T[3] = -1.0
    u[7] = 1.5
    z[11, 17] = np.nan
    for method in ("multinomial", "gumbel"):
        ids, o = _check_draft(z, T, u, method, 5, 0, "f32", f"bad rows {method}")
        assert ids[3] == -1 and ids[11] == -1
        assert (ids[7] == -1) == (method == "multinomial")
    x = W.config("verify64")
    z = x.draft.reshape(-1, x.V)
    T = np.repeat(x.temperature, x.gamma).astype(np.float32)
    u = x.uniforms[:, :x.gamma].reshape(-1).copy()
    for method in ("multinomial", "gumbel"):
        _check_draft(z, T, u, method, 2026, 1, "bf16", f"verify64 rows {method}")


@pytest.mark.parametrize("C", [None, 8])
def test_draft_sample_nonfinite_rows(C):
    """NaN and +inf anywhere in a row (first and last index, a middle
    segment), rows that are all -inf, and -inf entries in valid rows, with
    good rows after each bad one: flags and draws against the oracle, the
    greedy rows included."""
    V = 40000
    z, T, u = _draft_rows(V, "f32", 2, 6200, B=14)
    n = z.shape[0]
    z[1, 0] = np.nan
    z[4, V - 1] = np.inf
    z[8, V // 2 + 3] = np.nan
    z[10, :] = -np.inf
    z[13, 5000:9000] = -np.inf
    z[16, 123] = np.inf
    z[16, 124] = -np.inf
    z[19, ::7] = -np.inf
    z[22, 37] = np.nan
    T[22] = 0.0
    z[n - 1, V - 2] = np.nan
    with tune(cluster_size=C):
        for method in ("multinomial", "gumbel"):
            ids, o = _check_draft(z, T, u, method, 17, 3, "f32", f"nonfinite rows {method} C={C}")
            for r in (1, 4, 8, 10, 16, 22, n - 1):
                assert ids[r] == -1, (method, r, ids[r])
            for r in (13, 19):
                assert ids[r] >= 0 and np.isfinite(z[r, ids[r]]), (method, r, ids[r])


@pytest.mark.parametrize("C", [None, 2])
def test_draft_sample_gumbel_cold(C):
    """Low temperatures (T = 0.01 to 0.05) scale the keys up to |z k| ~ 10^4
    and make the per-chunk key bounds of the one-pass draw tight: draws
    against the oracle."""
    z, T, u = _draft_rows(65536, "f32", 1, 6300, B=12)
    T[:] = np.linspace(0.01, 0.05, T.size).astype(np.float32)
    with tune(cluster_size=C):
        ids, o = _check_draft(z, T, u, "gumbel", 31, 0, "f32", f"cold rows C={C}")
    assert np.all(ids >= 0)


def test_concurrent_calls_on_streams():
    """Verify, row statistics and Gumbel-max draft sampling launched back to
    back on three streams with no synchronisation between them (the library
    keeps no state between calls, so concurrent calls cannot interfere): each
    result matches the oracle."""
    import mtp_speculative_decoding_row_gb300 as mtp
    x = W.verify_inputs("conc", 16, 3, 40000, "bf16", 5300, family="sigma", sigmas=np.linspace(1.0, 6.0, 16),
                        delta=0.4, temperature=np.linspace(0.7, 1.2, 16))
    z, T, u = _draft_rows(30000, "bf16", 2, 6500, B=24)
    dv = [to_dev(a) for a in (x.target, x.draft, x.draft_ids, x.temperature, x.uniforms)]
    dz = [to_dev(a) for a in (z, T, u)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(3)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):  # several rounds in flight at once
        with torch.cuda.stream(streams[0]):
            v = mtp.mtp_rs_verify(*dv, stream=streams[0])
        with torch.cuda.stream(streams[1]):
            st = mtp.mtp_row_stats(dv[0], dv[1], dv[3], stream=streams[1])
        with torch.cuda.stream(streams[2]):
            ds = mtp.mtp_draft_sample(*dz, method="gumbel", seed=3, offset=1, stream=streams[2])
    torch.cuda.synchronize()
    g = {k: (t.cpu().numpy() if t is not None else None) for k, t in v._asdict().items()}
    o = oracle.verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms, want_stats=False)
    compare.assert_ok(compare.verify_report(g["tokens"], g["accept_len"], g["row_flags"], o, x.draft_ids, x.gamma,
                                            x.V, x.dtype, x=x), "concurrent verify")
    gs = {k: t.cpu().numpy() for k, t in st._asdict().items()}
    os_ = oracle.row_stats(x.target, x.draft, x.temperature)
    compare.assert_ok(compare.stats_report(gs["alpha"], gs["entropy"], os_, x.dtype, gs["row_flags"]),
                      "concurrent stats")
    od = oracle.draft_sample(z, T, u, method="gumbel", seed=3, offset=1)
    ids = ds.ids.cpu().numpy()
    np.testing.assert_array_equal(ds.row_flags.cpu().numpy(), od["flags"])
    assert not ((ids != od["ids"]) & ~(od["margin"] < compare.GUMBEL_MARGIN)).any()


def test_draft_sample_in_cuda_graph():
    """mtp_draft_sample, both draws, captured once in a CUDA graph on a side
    stream and replayed on two sets of rows copied into the captured buffers:
    each replay matches the oracle (the noise key and counter word are part
    of the captured launch)."""
    import mtp_speculative_decoding_row_gb300 as mtp
    sets = [_draft_rows(30000, "bf16", 2, 6400 + i, B=24) for i in range(2)]
    for method in ("multinomial", "gumbel"):
        bufs = [to_dev(a) for a in sets[0]]
        out = mtp.mtp_draft_sample(*bufs, method=method, seed=77, offset=5)  # plan caches before capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                mtp.mtp_draft_sample(*bufs, method=method, seed=77, offset=5, out=out, stream=s)
        torch.cuda.synchronize()
        for z, T, u in reversed(sets):
            for dst, src in zip(bufs, (z, T, u)):
                dst.copy_(to_dev(src))
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            ids, flags = out.ids.cpu().numpy(), out.row_flags.cpu().numpy()
            o = oracle.draft_sample(z, T, u, method=method, seed=77, offset=5)
            np.testing.assert_array_equal(flags, o["flags"], err_msg=method)
            lim = compare.GUMBEL_MARGIN if method == "gumbel" else compare.MARGIN
            bad = (ids != o["ids"]) & ~(o["margin"] < lim)
            assert not bad.any(), (method, np.nonzero(bad)[0][:8])


def test_draft_sample_gumbel_extreme_noise():
    """Noise at the top of the uniform's range.  With seed 4696 (offset 0),
    row 0, index 376 draws U = 1 - 2^-25, the largest Gumbel noise the
    generator gives (G = 17.33; the row's second largest is 8.64).  Single
    precision cannot hold that U; the noise must still come out right, not
    infinite: with a low logit at index 376 another index wins, with a
    moderately low one index 376 still wins."""
    seed, v_star = 4696, 376
    G = oracle.gumbel_noise(seed, 0, 0, 0, 0, 2048)
    assert int(np.argmax(G)) == v_star and G[v_star] == -np.log(-np.log1p(-2.0 ** -25))
    for z_star, wins in ((-12.0, False), (-8.5, True)):
        z = np.zeros((1, 2048), np.float32)
        z[0, v_star] = z_star
        T = np.ones(1, np.float32)
        u = np.full(1, 0.5, np.float32)
        ids, o = _check_draft(z, T, u, "gumbel", seed, 0, "f32", f"extreme noise z*={z_star}")
        assert (ids[0] == v_star) == wins, (ids, o["ids"])


# ------------------------------------------------------- diagnostics -------

def _logit_scale(x):
    t = W.bf16_bits_to_f32(x.target) if x.dtype == "bf16" else x.target
    d = W.bf16_bits_to_f32(x.draft) if x.dtype == "bf16" else x.draft
    T = np.where(x.temperature > 0, x.temperature, 1.0)[:, None]
    with np.errstate(invalid="ignore"):
        mt = np.nanmax(np.where(np.isfinite(t), np.abs(t), 0.0), axis=-1)[:, :x.gamma]
        md = np.nanmax(np.where(np.isfinite(d), np.abs(d), 0.0), axis=-1)
    return np.maximum(mt, md) / T


def _check_diag(x, what=""):
    import mtp_speculative_decoding_row_gb300 as mtp
    out = mtp.mtp_rs_diagnostics(to_dev(x.target), to_dev(x.draft), to_dev(x.temperature))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out._asdict().items()}
    o = oracle.diagnostics(x.target, x.draft, x.temperature)
    rep = compare.diag_report(g, o, x.dtype, _logit_scale(x))
    if rep["bad"]:
        raise AssertionError(f"{what} diagnostics parity failed: {rep}")
    return rep, g, o


DIAG_SWEEP = [
    # (V, dtype, gamma, C)
    (1024, "f32", 3, None),
    (4096, "bf16", 5, 4),
    (40000, "f32", 8, 16),
    (40000, "bf16", 7, 2),
    (30000, "f32", 2, 1),
    (64, "f32", 3, 16),
    (151936, "bf16", 3, None),
]


@pytest.mark.parametrize("V,dtype,gamma,C", DIAG_SWEEP)
def test_diagnostics(V, dtype, gamma, C):
    """alpha, H(p), H(q), KL(q || p), arg max draft, p(yhat) and the
    rejection-sampling-better test against the oracle; delta = 0 rows have
    q == p (alpha = 1, KL = 0); T = 0 and T < 0 rows are flagged."""
    B = 24
    T = np.linspace(0.5, 1.5, B).astype(np.float32)
    T[5] = 0.0
    T[11] = -1.0
    x = W.verify_inputs(f"diag{V}", B, gamma, V, dtype, 4000 + V + gamma, family="sigma",
                        sigmas=np.linspace(0.3, 8.0, B), delta=np.linspace(0.0, 1.5, B), temperature=T)
    with tune(cluster_size=C):
        rep, g, o = _check_diag(x, f"V={V} {dtype} gamma={gamma} C={C}")
    good = o["flags"] == 0
    assert good.sum() == B - 2
    np.testing.assert_array_equal(g["row_flags"][[5, 11]], [4, 4])
    # both outcomes of the boundary test occur
    assert (o["rs_better"][good] == 1).any() and (o["rs_better"][good] == 0).any()
    # q == p: alpha 1 and KL 0
    np.testing.assert_allclose(g["alpha"][0], 1.0, rtol=0, atol=2e-6)
    np.testing.assert_allclose(g["kl"][0], 0.0, rtol=0, atol=2e-6)


def test_diagnostics_masked_and_bad_logits():
    """-inf logits (masked vocabulary): p = 0 < q gives KL = inf, both -inf
    adds nothing; a NaN logit flags the row."""
    B, gamma, V = 6, 3, 8192
    x = W.verify_inputs("diagmask", B, gamma, V, "f32", 4100, family="sigma", sigmas=np.linspace(1, 4, B),
                        delta=0.4)
    x.target[0, 1, 100:300] = -np.inf          # p = 0 where q > 0: KL infinite
    x.target[1, :, 7000:] = -np.inf            # both masked: finite statistics
    x.draft[1, :, 7000:] = -np.inf
    x.target[2, 3, 5] = np.nan                 # H(p_gamma) row: flagged
    x.draft[3, 0, 17] = np.nan
    x.draft[4, 2, :] = -np.inf                 # all -inf draft row: flagged
    rep, g, o = _check_diag(x, "masked")
    assert np.isinf(o["kl"][0, 1]) and np.isinf(g["kl"][0, 1])
    assert np.all(np.isfinite(g["kl"][1]))
    np.testing.assert_array_equal(o["flags"][[2, 3, 4]], [1, 1, 1])


def test_diagnostics_full_config():
    """The deep256 workload (B = 256, gamma = 7, V = 151936, f32)."""
    x = W.config("deep256")
    rep, g, o = _check_diag(x, "deep256")
    # positions within 1e-5 of the boundary (an oracle-only count) stay rare
    assert rep["near_margin"] <= 0.05 * x.B * x.gamma


# ------------------------------------------------------------ flags --------

def test_flags_and_defined_outputs():
    x = W.verify_inputs("flags", 8, 3, 3000, "f32", 31, family="sigma", sigmas=2.0, delta=0.3)
    x.temperature[1] = -1.0  # 0 is greedy decoding; a negative temperature is invalid
    x.draft_ids[2, 1] = 3000
    x.uniforms[3, 2] = 1.0
    x.target[4, 0, 17] = np.nan
    x.draft[5, 0, :] = -np.inf
    x.target[6, 0, 5] = np.inf
    x.uniforms[7, 0] = np.nan
    for stats in (False, True):
        g = run_verify(x, stats)
        o = oracle.verify(x.target, x.draft, x.draft_ids, x.temperature, x.uniforms, want_stats=stats)
        np.testing.assert_array_equal(g["row_flags"], o["flags"])
        for b in range(1, 8):
            assert g["accept_len"][b] == -1 and np.all(g["tokens"][b] == -1)
        if stats:
            assert np.all(np.isnan(g["alpha"][1:])) and np.all(np.isnan(g["entropy"][1:]))


def test_masked_vocab_is_allowed():
    """-inf logits are probability 0, not an error."""
    x = W.verify_inputs("mask", 8, 3, 2048, "bf16", 32, family="sigma", sigmas=2.0, delta=0.3)
    x.target[:, :, 1000:1500] = W.to_bf16_bits(np.array([-np.inf], np.float32))[0]
    x.draft[:, :, 1200:1800] = W.to_bf16_bits(np.array([-np.inf], np.float32))[0]
    for stats in (False, True):
        rep, g, o = _check_verify(x, stats, "masked")
        assert np.all(g["row_flags"] == 0)


# ------------------------------------------------------------- TV loss -----

TV_SWEEP = [
    # (N, gamma, V, dtype, T, scale, C, nres cap)
    (6, 1, 1000, "f32", 1.0, 1.0, None, None),
    (6, 3, 4097, "bf16", 0.7, 0.5, 4, None),
    (5, 3, 40000, "bf16", 1.0, 1.0, 16, None),
    (4, 5, 12000, "f32", 1.3, 2.0, 8, 2),
    (4, 3, 7, "bf16", 1.0, 1.0, 2, 1),
    (3, 7, 151936, "bf16", 1.0, 1.0, None, None),
]


@pytest.mark.parametrize("kernel", [None, "stream"])
@pytest.mark.parametrize("N,gamma,V,dtype,T,scale,C,nres", TV_SWEEP)
def test_tv_loss(N, gamma, V, dtype, T, scale, C, nres, kernel):
    """The sweep on the planner's kernel (TMEM-resident where a position's
    draft rows fit in tensor memory, else streaming where rows are whole
    vectors and gamma <= 8, else cluster-resident) and on the streaming
    kernel."""
    x = W.tvloss_inputs("tv", N, gamma, V, dtype, 500 + V + gamma, delta=0.5, sigmas=np.linspace(1.0, 8.0, N))
    with tune(cluster_size=C, tv_resident_drafts=nres, tv_kernel=kcode(kernel)):
        out = run_tv(to_dev(x.target), to_dev(x.draft), T, scale)
    o = oracle.tv_loss(x.target, x.draft, T, scale)
    tf = W.bf16_bits_to_f32(x.target).astype(np.float64) if dtype == "bf16" else x.target.astype(np.float64)
    df = W.bf16_bits_to_f32(x.draft).astype(np.float64) if dtype == "bf16" else x.draft.astype(np.float64)
    rep = compare.tv_report(out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy(),
                            out.row_flags.cpu().numpy(), o, dtype, tf, df, T)
    compare.assert_ok(rep, f"tv N={N} V={V}")


def _random_tv_configs(n, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = "bf16" if rng.random() < 0.6 else "f32"
        V = int(rng.choice([int(rng.integers(2, 64)), int(rng.integers(64, 5000)), int(rng.integers(5000, 50000))]))
        out.append((i, dtype, V, int(rng.integers(1, 10)), int(rng.integers(1, 13))))
    return out


@pytest.mark.parametrize("i,dtype,V,N,gamma", _random_tv_configs(12))
def test_tv_loss_randomized_shapes(i, dtype, V, N, gamma):
    """Seeded random shapes for the TV loss forward and backward (V from 2 to
    50,000 with unaligned sizes, N up to 9, gamma up to 12: past the
    streaming limit of 8 the cluster-resident kernel runs), random
    temperature and gradient scale: loss, alpha and gradient against the
    oracle."""
    rng = np.random.default_rng(9500 + i)
    T, scale = float(rng.uniform(0.5, 1.5)), float(rng.uniform(0.1, 2.0))
    x = W.tvloss_inputs(f"tvr{i}", N, gamma, V, dtype, 9600 + i, delta=float(rng.uniform(0.1, 1.0)),
                        sigmas=rng.uniform(0.3, 9.0, N))
    out = run_tv(to_dev(x.target), to_dev(x.draft), T, scale)
    o = oracle.tv_loss(x.target, x.draft, T, scale)
    tf = W.bf16_bits_to_f32(x.target).astype(np.float64) if dtype == "bf16" else x.target.astype(np.float64)
    df = W.bf16_bits_to_f32(x.draft).astype(np.float64) if dtype == "bf16" else x.draft.astype(np.float64)
    rep = compare.tv_report(out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy(),
                            out.row_flags.cpu().numpy(), o, dtype, tf, df, T)
    compare.assert_ok(rep, f"random tv {i}: {dtype} V={V} N={N} gamma={gamma}")


def test_tv_loss_in_cuda_graph():
    """mtp_tv_loss_fwd_bwd captured once in a CUDA graph on a side stream and
    replayed on two input sets copied into the captured buffers: loss, alpha
    and gradient match the oracle for each set."""
    import mtp_speculative_decoding_row_gb300 as mtp
    T, scale = 0.9, 0.5
    xs = [W.tvloss_inputs(f"tvg{i}", 6, 3, 40000, "bf16", 640 + i, delta=0.5, sigmas=np.linspace(1.0, 8.0, 6))
          for i in range(2)]
    bufs = [to_dev(xs[0].target), to_dev(xs[0].draft)]
    out = mtp.mtp_tv_loss_fwd_bwd(*bufs, T, scale)  # plan caches and outputs before capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            mtp.mtp_tv_loss_fwd_bwd(*bufs, T, scale, out=out, stream=s)
    torch.cuda.synchronize()
    for x in reversed(xs):
        bufs[0].copy_(to_dev(x.target))
        bufs[1].copy_(to_dev(x.draft))
        out.grad.fill_(float("nan"))  # every entry must be rewritten by the replay
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        o = oracle.tv_loss(x.target, x.draft, T, scale)
        tf = W.bf16_bits_to_f32(x.target).astype(np.float64)
        df = W.bf16_bits_to_f32(x.draft).astype(np.float64)
        rep = compare.tv_report(out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy(),
                                out.row_flags.cpu().numpy(), o, "bf16", tf, df, T)
        compare.assert_ok(rep, "tv graph replay")


@pytest.mark.parametrize("N,gamma,V,dtype,C,clusters,ring,kernel", [
    (9, 3, 40000, "bf16", 16, 2, None, None),     # several positions per cluster: both exchange banks
    (7, 2, 20000, "f32", 4, 3, 3, None),
    (5, 4, 65536, "bf16", 8, 1, 2, None),
    (6, 3, 40000, "bf16", None, None, None, "resident"),
    (4, 5, 12000, "f32", 8, None, None, "resident"),
    (3, 8, 30000, "bf16", None, 2, None, None),   # gamma = 8, the streaming limit
    (3, 9, 30000, "bf16", None, None, None, None),  # gamma = 9 takes the resident kernel
    (9, 3, 40000, "bf16", 16, 2, None, "stream"),
    (7, 2, 20000, "f32", 4, 3, 3, "stream"),
    (3, 8, 30000, "bf16", None, 2, None, "stream"),
    # TMEM-resident kernel: cluster sizes, rings, several positions per cluster, the largest row per lane
    (11, 3, 151936, "bf16", 8, 3, 2, "tmem"),
    (9, 3, 151936, "bf16", None, None, 3, "tmem"),
    (8, 1, 50000, "f32", 8, 2, None, "tmem"),
    (10, 2, 60000, "f32", 8, 3, 4, "tmem"),
    (7, 4, 30000, "bf16", 4, 2, None, "tmem"),
    (6, 8, 16384, "f32", 8, 2, None, "tmem"),
    (13, 3, 4096, "bf16", 1, 4, 2, "tmem"),
    (5, 2, 8, "bf16", 2, None, None, "tmem"),     # V = 8: most warps hold no vector
])
def test_tv_loss_kernels(N, gamma, V, dtype, C, clusters, ring, kernel):
    """TMEM-resident, streaming and cluster-resident TV kernels, several
    positions per cluster (both exchange banks), ring depths, cluster sizes
    and the gamma limit."""
    x = W.tvloss_inputs("tvk", N, gamma, V, dtype, 600 + V + gamma, delta=0.5, sigmas=np.linspace(0.7, 9.0, N))
    with tune(cluster_size=C, max_clusters=clusters, ring_slots=ring, tv_kernel=kcode(kernel)):
        out = run_tv(to_dev(x.target), to_dev(x.draft), 0.8, 1.5)
    o = oracle.tv_loss(x.target, x.draft, 0.8, 1.5)
    tf = W.bf16_bits_to_f32(x.target).astype(np.float64) if dtype == "bf16" else x.target.astype(np.float64)
    df = W.bf16_bits_to_f32(x.draft).astype(np.float64) if dtype == "bf16" else x.draft.astype(np.float64)
    rep = compare.tv_report(out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy(),
                            out.row_flags.cpu().numpy(), o, dtype, tf, df, 0.8)
    compare.assert_ok(rep, f"tv kernels N={N} gamma={gamma} V={V} C={C} kernel={kernel}")


TV_VARIANTS = [
    # (N, gamma, V, dtype, shared, clamp_tau, C, kernel)
    (7, 3, 4096, "f32", True, None, None, None),
    (9, 3, 40000, "bf16", True, None, 16, None),
    (6, 5, 12000, "bf16", True, 0.5, 4, None),
    (6, 3, 30000, "f32", False, 0.3, None, None),
    (5, 2, 20000, "bf16", False, 1.0, 8, None),
    (5, 3, 4097, "bf16", True, 0.4, None, None),      # unaligned rows: the resident kernel
    (6, 3, 20000, "f32", True, 0.3, 4, "resident"),
    (4, 9, 8192, "bf16", True, None, None, None),     # gamma = 9: the resident kernel
    (9, 3, 40000, "bf16", True, None, 8, "tmem"),
    (6, 3, 30000, "f32", False, 0.3, None, "tmem"),
    (9, 3, 151936, "bf16", True, 0.4, 8, "tmem"),
]


@pytest.mark.parametrize("N,gamma,V,dtype,shared,tau,C,kernel", TV_VARIANTS)
def test_tv_loss_variants(N, gamma, V, dtype, shared, tau, C, kernel):
    """Shared target rows [N + gamma - 1, V] (pair (t, k) on row t + k) and
    the App. F clamped per-step loss, on both TV kernels."""
    if shared:
        x = W.tvloss_shared_inputs("tvs", N, gamma, V, dtype, 700 + V + gamma, delta=0.5,
                                   sigmas=np.linspace(0.7, 8.0, N + gamma - 1))
    else:
        x = W.tvloss_inputs("tvc", N, gamma, V, dtype, 700 + V + gamma, delta=0.5, sigmas=np.linspace(0.7, 8.0, N))
    import mtp_speculative_decoding_row_gb300 as mtp
    if tau is not None and tau < 1.0:
        # tau_max at the median step of the oracle's 1 - alpha: both sides of the clamp occur
        steps = np.sort(1 - oracle.tv_loss(x.target, x.draft, 0.9, 1.0, with_grad=False,
                                           shared_target=shared)["alpha"].ravel())
        mid = len(steps) // 2
        tau = float(0.5 * (steps[mid - 1] + steps[mid]))
    with tune(cluster_size=C, tv_kernel=kcode(kernel)):
        out = mtp.mtp_tv_loss_fwd_bwd(to_dev(x.target), to_dev(x.draft), 0.9, 1.25, shared_target=shared,
                                      clamp_tau=tau)
        torch.cuda.synchronize()
    o = oracle.tv_loss(x.target, x.draft, 0.9, 1.25, shared_target=shared, clamp_tau=tau)
    tf = W.bf16_bits_to_f32(x.target).astype(np.float64) if dtype == "bf16" else x.target.astype(np.float64)
    df = W.bf16_bits_to_f32(x.draft).astype(np.float64) if dtype == "bf16" else x.draft.astype(np.float64)
    if shared:
        tf = np.stack([tf[t:t + gamma] for t in range(N)])
    rep = compare.tv_report(out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy(),
                            out.row_flags.cpu().numpy(), o, dtype, tf, df, 0.9)
    compare.assert_ok(rep, f"tv variant N={N} gamma={gamma} V={V} shared={shared} tau={tau} kernel={kernel}")
    if tau is not None:
        steps = 1 - o["alpha"]
        assert ((steps > tau).any() and (steps < tau).any()) or tau >= 1.0
        assert np.min(np.abs(steps - tau)) > 1e-6  # no step on the kink


def _topk_of(x, K):
    """Top-K entries (values in storage dtype, int32 indices) of each target row."""
    tf = W.bf16_bits_to_f32(x.target) if x.dtype == "bf16" else x.target
    idx = np.argsort(-tf, axis=-1, kind="stable")[..., :K].astype(np.int32)
    return np.ascontiguousarray(np.take_along_axis(x.target, idx, axis=-1)), np.ascontiguousarray(idx)


@pytest.mark.parametrize("N,gamma,V,dtype,K,tau,C", [
    (5, 3, 4096, "f32", 16, None, None),
    (6, 3, 40000, "bf16", 64, None, 16),
    (4, 5, 12000, "bf16", 1, None, 4),
    (3, 8, 30000, "f32", 1000, 0.6, None),
    (4, 3, 151936, "bf16", 64, None, None),
])
def test_tv_loss_topk(N, gamma, V, dtype, K, tau, C):
    """Top-K target path (K cached target logits per pair, renormalised):
    loss, alpha and the full-row gradient against the oracle."""
    x = W.tvloss_inputs("tvk", N, gamma, V, dtype, 800 + V + K, delta=0.4, sigmas=np.linspace(0.8, 7.0, N))
    vals, idx = _topk_of(x, K)
    import mtp_speculative_decoding_row_gb300 as mtp
    with tune(cluster_size=C):
        out = mtp.mtp_tv_loss_topk(to_dev(vals), to_dev(idx), to_dev(x.draft), 0.9, 1.25, clamp_tau=tau)
        torch.cuda.synchronize()
    o = oracle.tv_loss_topk(vals, idx, x.draft, 0.9, 1.25, clamp_tau=tau)
    tf = W.bf16_bits_to_f32(x.target).astype(np.float64) if dtype == "bf16" else x.target.astype(np.float64)
    df = W.bf16_bits_to_f32(x.draft).astype(np.float64) if dtype == "bf16" else x.draft.astype(np.float64)
    masked = np.full_like(tf, -np.inf)
    np.put_along_axis(masked, idx.astype(np.int64), np.take_along_axis(tf, idx.astype(np.int64), axis=-1), axis=-1)
    rep = compare.tv_report(out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy(),
                            out.row_flags.cpu().numpy(), o, dtype, masked, df, 0.9)
    compare.assert_ok(rep, f"tv topk N={N} gamma={gamma} V={V} K={K}")


def test_tv_loss_topk_bad_index_and_nan():
    x = W.tvloss_inputs("tvkb", 5, 3, 8192, "f32", 880, delta=0.4, sigmas=np.linspace(1, 4, 5))
    vals, idx = _topk_of(x, 8)
    idx[1, 2, 3] = 8192
    vals[3, 0, 0] = np.nan
    x.draft[4, 1, 77] = np.inf
    import mtp_speculative_decoding_row_gb300 as mtp
    out = mtp.mtp_tv_loss_topk(to_dev(vals), to_dev(idx), to_dev(x.draft), 1.0, 1.0)
    torch.cuda.synchronize()
    o = oracle.tv_loss_topk(vals, idx, x.draft, 1.0, 1.0)
    np.testing.assert_array_equal(out.row_flags.cpu().numpy(), o["flags"])
    np.testing.assert_array_equal(o["flags"], [0, 2, 0, 1, 1])
    g = out.grad.cpu().numpy()
    assert np.all(g[[1, 3, 4]] == 0) and np.all(np.isnan(out.loss.cpu().numpy()[[1, 3, 4]]))


def test_tv_plan_kernels():
    """At the tvloss size the planner takes the TMEM-resident kernel: 4-CTA
    clusters whose gamma draft rows per position fit the CTAs' tensor
    memory, with shared memory above half of the SM's, so that a second CTA
    and its TMEM allocation never land on an SM."""
    import mtp_speculative_decoding_row_gb300 as mtp
    p = mtp.mtp_query_plan("tv_loss", "bf16", 16384, 3, 151936)
    assert p["cluster_size"] == 4 and p["resident_drafts"] == 3, p
    props = torch.cuda.get_device_properties(0)
    per_sm = props.shared_memory_per_multiprocessor
    assert per_sm // 2 < p["smem_bytes"] + 1024, p
    with tune(tv_kernel=kcode("stream")):
        s = mtp.mtp_query_plan("tv_loss", "bf16", 16384, 3, 151936)
    q = mtp.mtp_query_plan("tv_loss_resident", "bf16", 16384, 3, 151936)
    assert s["resident_drafts"] == 0 and q["resident_drafts"] >= 1
    assert s["clusters"] * s["cluster_size"] > q["clusters"] * q["cluster_size"]
    # gamma = 7 draft rows of a position do not fit in tensor memory: the request falls back to streaming
    with tune(tv_kernel=kcode("tmem")):
        f = mtp.mtp_query_plan("tv_loss", "bf16", 16384, 7, 151936)
    assert f["resident_drafts"] == 0, f


def test_tv_loss_tmem_wait_timeout():
    """Failure detection of the bounded waits, with no GPU fault: the
    cluster's first warp leaves out its first exchange record at position 4
    (test-only tuning fields), so every wait on that round gives up after
    20 ms.  The call returns; position 4 and the later positions of its
    cluster (positions 1, 4, 7, 10 belong to cluster 1 of 3) come back
    flagged MTP_ROW_TIMEOUT with a NaN loss and alpha and a zero gradient;
    every other position matches the oracle; and the next call, without the
    fault, is correct again."""
    import mtp_speculative_decoding_row_gb300 as mtp
    N, gamma, V = 12, 3, 40000
    x = W.tvloss_inputs("tvto", N, gamma, V, "bf16", 990, delta=0.5, sigmas=np.linspace(0.7, 6.0, N))
    T, scale = 0.9, 1.3
    with tune(tv_kernel=kcode("tmem"), max_clusters=3):
        assert mtp.mtp_query_plan("tv_loss", "bf16", N, gamma, V)["clusters"] == 3
        with tune(fault_wait_us=20000, fault_skip_position=4 + 1):
            out = run_tv(to_dev(x.target), to_dev(x.draft), T, scale)
        flags = out.row_flags.cpu().numpy()
        with pytest.raises(mtp.MTPError) as e:
            mtp.check_row_flags(out.row_flags)
        assert e.value.status == mtp.MTP_ERR_TIMEOUT
        again = run_tv(to_dev(x.target), to_dev(x.draft), T, scale)
    timed_out = np.array([4, 7, 10])
    assert list(np.nonzero(flags)[0]) == list(timed_out) and np.all(flags[timed_out] == mtp.ROW_TIMEOUT)
    loss, alpha, grad = out.loss.cpu().numpy(), out.alpha.cpu().numpy(), out.grad.cpu().numpy()
    assert np.all(np.isnan(loss[timed_out])) and np.all(np.isnan(alpha[timed_out]))
    assert np.all(grad[timed_out] == 0)
    o = oracle.tv_loss(x.target, x.draft, T, scale)
    ok = np.setdiff1d(np.arange(N), timed_out)
    tf = W.bf16_bits_to_f32(x.target).astype(np.float64)
    df = W.bf16_bits_to_f32(x.draft).astype(np.float64)
    sub = {k: (v[ok] if isinstance(v, np.ndarray) and v.shape[:1] == (N,) else v) for k, v in o.items()}
    rep = compare.tv_report(loss[ok], alpha[ok], grad[ok], flags[ok], sub, "bf16", tf[ok], df[ok], T)
    compare.assert_ok(rep, "positions outside the timed-out cluster")
    rep = compare.tv_report(again.loss.cpu().numpy(), again.alpha.cpu().numpy(), again.grad.cpu().numpy(),
                            again.row_flags.cpu().numpy(), o, "bf16", tf, df, T)
    compare.assert_ok(rep, "the call after the timeout")


def test_tv_loss_full_config_sampled():
    """N = 16,384, gamma = 3, V = 151,936 bf16 on device: sampled positions
    against the oracle, sum_j grad = 0 on every row, loss in [-gamma, 0]."""
    x = W.config("tvloss", device="cuda")
    out = run_tv(x.target, x.draft, x.temperature, x.grad_scale)
    loss = out.loss.cpu().numpy()
    assert np.all(out.row_flags.cpu().numpy() == 0)
    assert np.all(loss <= 0) and np.all(loss >= -x.gamma)
    rows = out.grad.view(-1, x.V)
    sums = torch.zeros(rows.shape[0], dtype=torch.float64, device="cuda")
    for s in range(0, rows.shape[0], 4096):
        sums[s:s + 4096] = rows[s:s + 4096].double().sum(dim=1)
    # per-element bar is 1e-4; fp32 normalisers (log2 Z ~ 17) give ~1e-6 relative error in every q
    assert sums.abs().max().item() < 1e-4
    idx = np.unique(np.linspace(0, x.N - 1, 24).astype(int))
    it = torch.from_numpy(idx).cuda()
    tb, db = to_host_bits(x.target[it]), to_host_bits(x.draft[it])
    o = oracle.tv_loss(tb, db, x.temperature, x.grad_scale)
    rep = compare.tv_report(loss[idx], out.alpha[it].cpu().numpy(), out.grad[it].cpu().numpy(),
                            out.row_flags[it].cpu().numpy(), o, "bf16",
                            W.bf16_bits_to_f32(tb).astype(np.float64), W.bf16_bits_to_f32(db).astype(np.float64),
                            x.temperature)
    compare.assert_ok(rep, "tvloss sampled")
    print("tvloss sampled", {k: v for k, v in rep.items() if not isinstance(v, list)})


@pytest.mark.parametrize("kernel", [None, "stream", "resident"])
def test_tv_loss_bad_temperature_and_nan(kernel):
    x = W.tvloss_inputs("tvbad", 3, 2, 2000, "f32", 9, sigmas=2.0)
    x.target[1, 1, 3] = np.nan
    with tune(tv_kernel=kcode(kernel), max_clusters=1 if kernel != "resident" else None):
        out = run_tv(to_dev(x.target), to_dev(x.draft), 1.0, 1.0)
    f = out.row_flags.cpu().numpy()
    assert list(f) == [0, oracle.ROW_NONFINITE, 0]
    o = oracle.tv_loss(x.target, x.draft, 1.0, 1.0)
    np.testing.assert_allclose(out.loss.cpu().numpy()[[0, 2]], o["loss"][[0, 2]], rtol=1e-5)
    assert np.isnan(out.loss[1].item()) and torch.all(out.grad[1] == 0)
    with tune(tv_kernel=kcode(kernel)):
        out = run_tv(to_dev(x.target), to_dev(x.draft), 0.0, 1.0)
    assert np.all(out.row_flags.cpu().numpy() == oracle.ROW_BAD_TEMP)
    assert torch.all(out.grad == 0)
