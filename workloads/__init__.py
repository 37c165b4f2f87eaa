"""Seeded synthetic inputs for MTP verification, row statistics and the TV loss.

This module only draws numbers: logits, draft ids, temperatures and uniforms.
It holds none of the method's arithmetic (no softmax, no overlap, entropy or
CDF) and it is the one module that both the CUDA path's harness and the CPU
oracle's tests take their inputs from.

Recipe (all draws from NumPy ``Philox``; config index ``c``):

* uniforms: ``Philox(c)``, ``random(dtype=float32)`` so every value lies in
  [0, 1) exactly; ``u[b, 0..gamma-1]`` are the accept tests, ``u[b, gamma]``
  the final draw.
* target logits: seed ``100 + c``, one child stream per sequence, standard
  normal draws scaled per row; rounded to bfloat16 (nearest-even) where the
  workload is bf16.
* draft logits: the *rounded* target plus ``delta_b * N(0, 1)`` from seed
  ``200 + c``, rounded again.
* draft ids: a sample from ``q = softmax(draft / T_b)`` per draft row, drawn
  with the Gumbel-max construction ``argmax_v(draft_v / T_b + G_v)`` in float64
  from seed ``300 + c``.  This stands in for the draft stage that precedes
  verification; the verify path itself never draws Gumbel noise.
* per-row parameters (temperatures, mismatch, row families): seed ``400 + c``.

Entropy-spanning rows use ``z = sigma_b * g`` with ``sigma_b`` geometric between
``SIGMA_H4`` and ``SIGMA_H05``.  Over 64 standard-normal reference rows at
V = 151,936 and T = 1 the median entropy of softmax(sigma * g) is about
4.1 nats at sigma = 4.7 and about 0.48 nats at sigma = 14, so the schedule
spans the 0.5-4 nat range the pages study (rows in this regime scatter widely
around the median; the test suite checks the span with the oracle).

The pages' own workloads (Math, Code, SWE, Agent and MT-Bench rollouts of
trained models) are not available; these rows stand in for them.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

V_QWEN = 151936  # full vocabulary size of the pages' models

SIGMA_H4 = 4.75   # median H(softmax(sigma g)) ~ 4 nats at V = 151,936
SIGMA_H05 = 14.0  # median H ~ 0.5 nats


def philox(*key: int) -> np.random.Generator:
    """A Philox-4x64 generator keyed by a tuple of non-negative ints."""
    if len(key) == 1:
        return np.random.Generator(np.random.Philox(key[0]))
    return np.random.Generator(np.random.Philox(np.random.SeedSequence(list(key))))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def entropy_span_sigmas(n: int) -> np.ndarray:
    """n scales, geometric from SIGMA_H4 (about 4 nats) to SIGMA_H05 (0.5)."""
    if n == 1:
        return np.array([SIGMA_H4])
    f = np.arange(n) / (n - 1)
    return SIGMA_H4 * (SIGMA_H05 / SIGMA_H4) ** f


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


@dataclass
class VerifyInputs:
    """Inputs of one batched verify call (host arrays).

    target  [B, gamma+1, V] float32, or uint16 bfloat16 bit patterns
    draft   [B, gamma,   V] same storage as target
    draft_ids [B, gamma] int32, temperature [B] float32, uniforms [B, gamma+1]
    float32.
    """

    name: str
    B: int
    gamma: int
    V: int
    dtype: str  # "f32" or "bf16"
    target: np.ndarray
    draft: np.ndarray
    draft_ids: np.ndarray
    temperature: np.ndarray
    uniforms: np.ndarray
    want_stats: bool = False
    meta: dict = field(default_factory=dict)

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logits_f32(self, which: str) -> np.ndarray:
        a = getattr(self, which)
        return bf16_bits_to_f32(a) if self.dtype == "bf16" else a


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def _widen(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x) if dtype == "bf16" else x


def _zipf_row(rng: np.random.Generator, V: int, s: float = 1.1, peak: float = 8.0) -> np.ndarray:
    """Peaked Zipf-like logits: rank r gets -s ln r under a random permutation,
    and the rank-1 token gets +peak."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    z = (-s * np.log(ranks)).astype(np.float32)
    z[0] += peak
    out = np.empty(V, dtype=np.float32)
    out[rng.permutation(V)] = z
    return out


def verify_inputs(
    name: str,
    B: int,
    gamma: int,
    V: int,
    dtype: str,
    c: int,
    *,
    family: str = "entropy_span",
    sigmas=None,
    delta=0.3,
    temperature=1.0,
    high_entropy_frac: float = 0.3,
    want_stats: bool = False,
) -> VerifyInputs:
    """Draw one verify workload.

    family: "sigma" (per-sequence scales from ``sigmas``), "entropy_span"
    (geometric schedule over sequences) or "rl_mix" (per target row: with
    probability ``high_entropy_frac`` N(0, 1), else a peaked Zipf(1.1) row).
    delta, temperature: scalars or per-sequence arrays.
    """
    assert dtype in ("f32", "bf16") and B >= 0 and gamma >= 1 and V >= 1
    prm = philox(400 + c)
    if family == "sigma":
        sig = np.broadcast_to(np.asarray(sigmas, dtype=np.float64), (B,)).copy()
    elif family == "entropy_span":
        sig = entropy_span_sigmas(B)
    elif family == "rl_mix":
        sig = np.ones(B)
        high = prm.random((B, gamma + 1)) < high_entropy_frac
    else:
        raise ValueError(family)
    delta = np.broadcast_to(np.asarray(delta, dtype=np.float64), (B,)).copy()
    temp = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)).copy()

    esz = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((B, gamma + 1, V), dtype=esz)
    draft = np.empty((B, gamma, V), dtype=esz)
    ids = np.empty((B, gamma), dtype=np.int32)

    def one(b: int) -> None:
        tr = philox(100 + c, b)
        if family == "rl_mix":
            rows = []
            for i in range(gamma + 1):
                if high[b, i]:
                    rows.append(tr.standard_normal(V, dtype=np.float32))
                else:
                    rows.append(_zipf_row(tr, V))
            z = np.stack(rows)
        else:
            z = tr.standard_normal((gamma + 1, V), dtype=np.float32) * np.float32(sig[b])
        target[b] = _round(z, dtype)
        zt = _widen(target[b, :gamma], dtype)
        nz = philox(200 + c, b).standard_normal((gamma, V), dtype=np.float32)
        draft[b] = _round(zt + np.float32(delta[b]) * nz, dtype)
        # Draft-stage sample y ~ softmax(draft / T) by Gumbel-max (float64);
        # at T = 0 (greedy) the draft's arg max.
        u = philox(300 + c, b).random((gamma, V))
        if temp[b] > 0:
            dz = _widen(draft[b], dtype).astype(np.float64) / float(temp[b])
            with np.errstate(divide="ignore"):
                gum = -np.log(-np.log(u))
            ids[b] = np.argmax(dz + gum, axis=1).astype(np.int32)
        else:
            ids[b] = np.argmax(_widen(draft[b], dtype), axis=1).astype(np.int32)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(B)))

    uniforms = philox(c).random((B, gamma + 1), dtype=np.float32)
    meta = {"family": family, "sigma": sig, "delta": delta}
    if family == "rl_mix":
        meta["high_entropy_rows"] = high
    return VerifyInputs(name, B, gamma, V, dtype, target, draft, ids, temp, uniforms, want_stats, meta)


@dataclass
class TVLossInputs:
    """Inputs of one TV-loss call: target, draft [N, gamma, V] (float32 or
    bf16 bits), one temperature and the gradient scale."""

    name: str
    N: int
    gamma: int
    V: int
    dtype: str
    target: object  # np.ndarray on the host, or a device tensor
    draft: object
    temperature: float
    grad_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4


def tvloss_inputs(name: str, N: int, gamma: int, V: int, dtype: str, c: int, *, delta: float = 0.5,
                  temperature: float = 1.0, grad_scale: float = 1.0, sigmas=None) -> TVLossInputs:
    """Host (NumPy) TV-loss inputs: per position t, target rows
    sigma_t * N(0, 1) (entropy-spanning unless ``sigmas`` is given) and draft
    = rounded target + delta * N(0, 1)."""
    sig = entropy_span_sigmas(N) if sigmas is None else np.broadcast_to(np.asarray(sigmas, np.float64), (N,))
    esz = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((N, gamma, V), dtype=esz)
    draft = np.empty((N, gamma, V), dtype=esz)

    def one(t: int) -> None:
        z = philox(100 + c, t).standard_normal((gamma, V), dtype=np.float32) * np.float32(sig[t])
        target[t] = _round(z, dtype)
        nz = philox(200 + c, t).standard_normal((gamma, V), dtype=np.float32)
        draft[t] = _round(_widen(target[t], dtype) + np.float32(delta) * nz, dtype)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(N)))
    return TVLossInputs(name, N, gamma, V, dtype, target, draft, float(temperature), float(grad_scale),
                        {"sigma": np.asarray(sig), "delta": delta, "backend": "numpy"})


def tvloss_inputs_device(name: str, N: int, gamma: int, V: int, c: int, device, *, delta: float = 0.5,
                         temperature: float = 1.0, grad_scale: float = 1.0, chunk: int = 512) -> TVLossInputs:
    """Device-resident bf16 TV-loss inputs for sizes too large to draw on the
    host (torch's seeded CUDA Philox, one generator per chunk of positions).
    Same recipe as :func:`tvloss_inputs`; the streams differ from NumPy's, so
    CPU checks copy the sampled positions' inputs back to the host."""
    import torch

    sig = entropy_span_sigmas(N)
    target = torch.empty((N, gamma, V), dtype=torch.bfloat16, device=device)
    draft = torch.empty((N, gamma, V), dtype=torch.bfloat16, device=device)
    sig_t = torch.tensor(sig, dtype=torch.float32, device=device)
    for s in range(0, N, chunk):
        e = min(N, s + chunk)
        g = torch.Generator(device=device)
        g.manual_seed((100 + c) * 1_000_003 + s)
        z = torch.randn((e - s, gamma, V), generator=g, device=device, dtype=torch.float32)
        z.mul_(sig_t[s:e, None, None])
        tb = z.to(torch.bfloat16)
        target[s:e] = tb
        g.manual_seed((200 + c) * 1_000_003 + s)
        torch.randn((e - s, gamma, V), generator=g, device=device, dtype=torch.float32, out=z)
        z.mul_(delta).add_(tb.float())
        draft[s:e] = z.to(torch.bfloat16)
        del z, tb
    return TVLossInputs(name, N, gamma, V, "bf16", target, draft, float(temperature), float(grad_scale),
                        {"sigma": sig, "delta": delta, "backend": "torch-cuda"})


def tvloss_shared_inputs(name: str, N: int, gamma: int, V: int, dtype: str, c: int, *, delta: float = 0.5,
                         temperature: float = 1.0, grad_scale: float = 1.0, sigmas=None) -> TVLossInputs:
    """Host TV-loss inputs in the shared-target layout: target rows r = 0 ..
    N + gamma - 2, sigma_r * N(0, 1) (entropy-spanning unless ``sigmas``
    gives one value per row), and draft[t, k] = rounded target row t + k +
    delta * N(0, 1).  ``target`` is [N + gamma - 1, V]."""
    R = N + gamma - 1
    sig = entropy_span_sigmas(R) if sigmas is None else np.broadcast_to(np.asarray(sigmas, np.float64), (R,))
    esz = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((R, V), dtype=esz)
    draft = np.empty((N, gamma, V), dtype=esz)
    for r in range(R):
        target[r] = _round(philox(100 + c, r).standard_normal(V, dtype=np.float32) * np.float32(sig[r]), dtype)

    def one(t: int) -> None:
        nz = philox(200 + c, t).standard_normal((gamma, V), dtype=np.float32)
        draft[t] = _round(_widen(target[t:t + gamma], dtype) + np.float32(delta) * nz, dtype)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(N)))
    return TVLossInputs(name, N, gamma, V, dtype, target, draft, float(temperature), float(grad_scale),
                        {"sigma": np.asarray(sig), "delta": delta, "backend": "numpy", "layout": "shared"})


def tvloss_shared_inputs_device(name: str, N: int, gamma: int, V: int, c: int, device, *, delta: float = 0.5,
                                temperature: float = 1.0, grad_scale: float = 1.0,
                                chunk: int = 512) -> TVLossInputs:
    """Device-resident bf16 inputs of :func:`tvloss_shared_inputs` for sizes
    too large for the host (torch's seeded CUDA Philox per chunk)."""
    import torch

    R = N + gamma - 1
    sig = entropy_span_sigmas(R)
    target = torch.empty((R, V), dtype=torch.bfloat16, device=device)
    draft = torch.empty((N, gamma, V), dtype=torch.bfloat16, device=device)
    sig_t = torch.tensor(sig, dtype=torch.float32, device=device)
    g = torch.Generator(device=device)
    for s in range(0, R, chunk):
        e = min(R, s + chunk)
        g.manual_seed((100 + c) * 1_000_003 + s)
        z = torch.randn((e - s, V), generator=g, device=device, dtype=torch.float32)
        target[s:e] = (z * sig_t[s:e, None]).to(torch.bfloat16)
        del z
    for s in range(0, N, chunk):
        e = min(N, s + chunk)
        g.manual_seed((200 + c) * 1_000_003 + s)
        z = torch.randn((e - s, gamma, V), generator=g, device=device, dtype=torch.float32)
        z.mul_(delta)
        for k in range(gamma):
            z[:, k].add_(target[s + k:e + k].float())
        draft[s:e] = z.to(torch.bfloat16)
        del z
    return TVLossInputs(name, N, gamma, V, "bf16", target, draft, float(temperature), float(grad_scale),
                        {"sigma": sig, "delta": delta, "backend": "torch-cuda", "layout": "shared"})


def subset(x: VerifyInputs, B: int) -> VerifyInputs:
    """The first B sequences of a verify workload (same rows and parameters)."""
    return VerifyInputs(x.name, B, x.gamma, x.V, x.dtype, x.target[:B], x.draft[:B], x.draft_ids[:B],
                        x.temperature[:B], x.uniforms[:B], x.want_stats, dict(x.meta))


# The five workloads: (index c, description).
CONFIG_NAMES = ["tiny", "verify64", "rl512", "deep256", "tvloss"]


def config(name: str, *, device=None, N_override: int | None = None):
    """Draw the named workload.

    tiny      B=4,   gamma=3, V=1024,    f32,  sigma_b in {0.5,1,2,4}, delta 0.3, T=1
    verify64  B=64,  gamma=3, V=151,936, bf16, entropy-spanning, delta 0.3, T=1
    rl512     B=512, gamma=3, V=151,936, bf16, 30% N(0,1) rows else peaked
              Zipf(1.1)+8; delta_b in {0.1,0.5}, T_b in {0.6,1.0}
    deep256   B=256, gamma=7, V=151,936, f32, entropy-spanning,
              delta_b = b/(B-1), T_b cycling {0.6,0.8,1.0}; with alpha and H
    tvloss    N=16,384, gamma=3, V=151,936, bf16, entropy-spanning,
              draft = target + N(0, 0.5), T=1, grad_scale=1
    """
    c = CONFIG_NAMES.index(name)
    if name == "tiny":
        return verify_inputs(name, 4, 3, 1024, "f32", c, family="sigma", sigmas=[0.5, 1.0, 2.0, 4.0], delta=0.3)
    if name == "verify64":
        return verify_inputs(name, 64, 3, V_QWEN, "bf16", c, family="entropy_span", delta=0.3)
    if name == "rl512":
        prm = philox(400 + c, 1)
        delta = np.where(prm.random(512) < 0.5, 0.1, 0.5)
        temp = np.where(prm.random(512) < 0.5, 0.6, 1.0).astype(np.float32)
        return verify_inputs(name, 512, 3, V_QWEN, "bf16", c, family="rl_mix", delta=delta, temperature=temp)
    if name == "deep256":
        B = 256
        delta = np.arange(B) / (B - 1)
        temp = np.array([0.6, 0.8, 1.0], dtype=np.float32)[np.arange(B) % 3]
        return verify_inputs(name, B, 7, V_QWEN, "f32", c, family="entropy_span", delta=delta, temperature=temp,
                             want_stats=True)
    if name == "tvloss":
        N = N_override or 16384
        if device is None:
            return tvloss_inputs(name, N, 3, V_QWEN, "bf16", c)
        return tvloss_inputs_device(name, N, 3, V_QWEN, c, device)
    raise ValueError(name)
