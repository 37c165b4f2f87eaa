"""Checks of the seeded input generators (CPU only)."""
import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
import workloads as W


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100_000).astype(np.float32) * 7
    x[:4] = [0.0, -0.0, 1e-40, 3.0e38]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(W.to_bf16_bits(x), ref)
    np.testing.assert_array_equal(W.bf16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_tiny_config_shapes_and_determinism():
    a = W.config("tiny")
    b = W.config("tiny")
    assert a.target.shape == (4, 4, 1024) and a.draft.shape == (4, 3, 1024) and a.target.dtype == np.float32
    assert a.draft_ids.dtype == np.int32 and a.draft_ids.min() >= 0 and a.draft_ids.max() < 1024
    assert a.uniforms.dtype == np.float32 and a.uniforms.min() >= 0 and a.uniforms.max() < 1
    np.testing.assert_array_equal(a.uniforms, np.random.Generator(np.random.Philox(0)).random((4, 4), np.float32))
    for k in ("target", "draft", "draft_ids", "uniforms", "temperature"):
        np.testing.assert_array_equal(getattr(a, k), getattr(b, k))


def test_draft_ids_are_samples_from_q():
    """Randomised probability-integral transform of the drawn ids under
    q = softmax(draft / T) is Uniform(0, 1) when ids ~ q."""
    B, V, T = 4000, 8, 0.7
    x = W.verify_inputs("pit", B, 1, V, "f32", 77, family="sigma", sigmas=1.5, delta=0.4, temperature=T)
    q = scipy.special.softmax(x.draft[:, 0].astype(np.float64) / T, axis=-1)
    y = x.draft_ids[:, 0]
    cdf_before = np.cumsum(q, axis=1)[np.arange(B), y] - q[np.arange(B), y]
    u = cdf_before + np.random.default_rng(5).random(B) * q[np.arange(B), y]
    assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3


def test_entropy_span_endpoints():
    """sigma endpoints give median entropies near 4 and 0.5 nats at V = 151,936."""
    n = 24
    for sig, lo, hi in ((W.SIGMA_H4, 3.4, 4.7), (W.SIGMA_H05, 0.25, 0.9)):
        x = W.verify_inputs("span", n, 1, W.V_QWEN, "bf16", 91, family="sigma", sigmas=sig)
        st = oracle.row_stats(x.target, x.draft, x.temperature)
        med = np.median(st["entropy"])
        assert lo < med < hi, (sig, med)


def test_rl_mix_rows():
    x = W.verify_inputs("rl", 8, 3, W.V_QWEN, "bf16", 2, family="rl_mix", delta=0.1, temperature=1.0)
    st = oracle.row_stats(x.target, x.draft, x.temperature)
    high = x.meta["high_entropy_rows"]
    assert high.any() and (~high).any()
    assert np.all(st["entropy"][high] > 10.5)
    assert np.all(st["entropy"][~high] < 0.2)
