"""Float64 CPU oracle (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It wraps ``mtp_oracle.c`` (plain C,
double precision, OpenMP over rows) through ctypes and shares nothing with the
CUDA library.  See ``mtp_oracle.c`` for the definitions it follows and the
pages' sections they come from.

Every function takes host arrays: logits as float32, float64 or uint16
bfloat16 bit patterns (widened exactly), and returns NumPy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mtp_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ROW_NONFINITE, ROW_BAD_ID, ROW_BAD_TEMP, ROW_ZERO_MASS, ROW_BAD_UNIFORM = 1, 2, 4, 8, 16
ERROR_BITS = ROW_NONFINITE | ROW_BAD_ID | ROW_BAD_TEMP | ROW_BAD_UNIFORM


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2 -fopenmp) if missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_softmax.argtypes = [P, I, I, I, D, P]
            lib.oracle_verify.argtypes = [P, P, I, P, P, P, I, I, I, I, P, P, P, P, P, P, P, P]
            lib.oracle_row_stats.argtypes = [P, P, I, P, I, I, I, P, P, P, P]
            lib.oracle_tv_loss.argtypes = [P, P, I, D, I, I, I, D, I, P, P, P, P, P, P]
            lib.oracle_tv_loss_ex.argtypes = [P, P, I, D, I, I, I, D, I, I, I, D, P, P, P, P, P, P]
            lib.oracle_to_verify.argtypes = [P, P, I, P, P, I, I, I, P, P, P, P, P, P]
            lib.oracle_diagnostics.argtypes = [P, P, I, P, I, I, I, P, P, P, P, P, P, P, P, P, P]
            U32 = ctypes.c_uint32
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_gumbel_noise.argtypes = [U32, U32, U32, U32, I, I, I, P]
            lib.oracle_gumbel_verify.argtypes = [P, P, I, P, P, P, U32, U32, U32, I, I, I, P, P, P, P, P]
            lib.oracle_tv_loss_topk.argtypes = [P, P, P, I, D, I, I, I, I, D, I, I, D, P, P, P, P, P, P]
            lib.oracle_draft_sample.argtypes = [P, I, P, P, I, U32, U32, U32, I, I, P, P, P]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_set_threads.argtypes = [I]
            lib.oracle_set_threads.restype = None
            for f in (lib.oracle_softmax, lib.oracle_verify, lib.oracle_row_stats, lib.oracle_tv_loss,
                      lib.oracle_num_threads):
                f.restype = I
            _lib = lib
    return _lib


def _logits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    if a.dtype == np.float64:
        return a, 2
    raise TypeError(f"unsupported logit storage {a.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads() -> int:
    """Threads the oracle's parallel loops use (OMP_NUM_THREADS respected)."""
    return _load().oracle_num_threads()


def set_threads(n: int) -> None:
    """Thread count of the oracle's later parallel loops (benchmark timing on a
    stated number of cores).  Results do not depend on it."""
    _load().oracle_set_threads(int(n))


def softmax(z, T: float = 1.0) -> np.ndarray:
    """p = softmax(z / T) along the last axis, float64."""
    z, dt = _logits(z)
    V = z.shape[-1]
    rows = z.size // V
    p = np.empty(z.shape, dtype=np.float64)
    _load().oracle_softmax(_ptr(z), dt, rows, V, float(T), _ptr(p))
    return p


def verify(target, draft, draft_ids, temperature, uniforms, want_stats: bool = False) -> dict:
    """Batched RS verification.  target [B, gamma+1, V], draft [B, gamma, V].

    Returns dict with tokens [B, gamma+1] int32 (-1 padded), accept_len [B],
    flags [B], acc_margin [B, gamma], cdf_margin [B], and with want_stats
    alpha, tv [B, gamma], entropy [B, gamma+1].
    """
    t, dt = _logits(target)
    d, dt2 = _logits(draft)
    assert dt == dt2
    B, g1, V = t.shape
    gamma = g1 - 1
    assert d.shape == (B, gamma, V)
    ids = np.ascontiguousarray(draft_ids, dtype=np.int32).reshape(B, gamma)
    temp = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, gamma + 1)
    out = {
        "tokens": np.empty((B, gamma + 1), np.int32),
        "accept_len": np.empty(B, np.int32),
        "flags": np.empty(B, np.int32),
        "acc_margin": np.empty((B, gamma), np.float64),
        "cdf_margin": np.empty(B, np.float64),
    }
    if want_stats:
        out["alpha"] = np.empty((B, gamma), np.float64)
        out["tv"] = np.empty((B, gamma), np.float64)
        out["entropy"] = np.empty((B, gamma + 1), np.float64)
    rc = _load().oracle_verify(
        _ptr(t), _ptr(d), dt, _ptr(ids), _ptr(temp), _ptr(u), B, gamma, V, int(want_stats),
        _ptr(out["tokens"]), _ptr(out["accept_len"]), _ptr(out.get("alpha")), _ptr(out.get("tv")),
        _ptr(out.get("entropy")), _ptr(out["flags"]), _ptr(out["acc_margin"]), _ptr(out["cdf_margin"]))
    if rc:
        raise RuntimeError(f"oracle_verify failed ({rc})")
    return out


def to_verify(target, draft, temperature, uniforms) -> dict:
    """Batched target-only verification: draft token = arg max of the draft
    logits, accepted iff u < p(y); replacement from p without y; T = 0 is
    greedy.  Returns tokens [B, gamma+1], accept_len [B], yhat [B, gamma]
    (-1 past the chain), flags [B], acc_margin [B, gamma] = |u - p(y)|,
    cdf_margin [B]."""
    t, dt = _logits(target)
    d, dt2 = _logits(draft)
    assert dt == dt2
    B, g1, V = t.shape
    gamma = g1 - 1
    assert d.shape == (B, gamma, V)
    temp = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, gamma + 1)
    out = {
        "tokens": np.empty((B, gamma + 1), np.int32),
        "accept_len": np.empty(B, np.int32),
        "yhat": np.empty((B, gamma), np.int32),
        "flags": np.empty(B, np.int32),
        "acc_margin": np.empty((B, gamma), np.float64),
        "cdf_margin": np.empty(B, np.float64),
    }
    rc = _load().oracle_to_verify(_ptr(t), _ptr(d), dt, _ptr(temp), _ptr(u), B, gamma, V, _ptr(out["tokens"]),
                                  _ptr(out["accept_len"]), _ptr(out["yhat"]), _ptr(out["flags"]),
                                  _ptr(out["acc_margin"]), _ptr(out["cdf_margin"]))
    if rc:
        raise RuntimeError(f"oracle_to_verify failed ({rc})")
    return out


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 of one 4-word counter under a 2-word key (uint32)."""
    c = np.ascontiguousarray(counter, dtype=np.uint32).reshape(4)
    k = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
    out = np.empty(4, np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def _seed_words(seed: int):
    seed = int(seed) & ((1 << 64) - 1)
    return seed & 0xFFFFFFFF, seed >> 32


def gumbel_noise(seed: int, offset: int, b: int, i: int, v0: int, n: int) -> np.ndarray:
    """Standard Gumbel noise G_v, v = v0 .. v0+n-1, of row i of sequence b."""
    lo, hi = _seed_words(seed)
    out = np.empty(n, np.float64)
    _load().oracle_gumbel_noise(lo, hi, int(offset) & 0xFFFFFFFF, int(b), int(i), int(v0), int(n), _ptr(out))
    return out


def gumbel_verify(target, draft, draft_ids, temperature, uniforms, seed: int, offset: int = 0) -> dict:
    """Batched verify whose final token (residual or bonus) is a Gumbel-max
    draw with Philox noise keyed by (seed, offset, sequence, row).  Returns
    tokens [B, gamma+1], accept_len [B], flags [B], acc_margin [B, gamma],
    gumbel_margin [B] (best minus second best key of the final draw)."""
    t, dt = _logits(target)
    d, dt2 = _logits(draft)
    assert dt == dt2
    B, g1, V = t.shape
    gamma = g1 - 1
    assert d.shape == (B, gamma, V)
    ids = np.ascontiguousarray(draft_ids, dtype=np.int32).reshape(B, gamma)
    temp = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, gamma + 1)
    lo, hi = _seed_words(seed)
    out = {
        "tokens": np.empty((B, gamma + 1), np.int32),
        "accept_len": np.empty(B, np.int32),
        "flags": np.empty(B, np.int32),
        "acc_margin": np.empty((B, gamma), np.float64),
        "gumbel_margin": np.empty(B, np.float64),
    }
    rc = _load().oracle_gumbel_verify(_ptr(t), _ptr(d), dt, _ptr(ids), _ptr(temp), _ptr(u), lo, hi,
                                      int(offset) & 0xFFFFFFFF, B, gamma, V, _ptr(out["tokens"]),
                                      _ptr(out["accept_len"]), _ptr(out["flags"]), _ptr(out["acc_margin"]),
                                      _ptr(out["gumbel_margin"]))
    if rc:
        raise RuntimeError(f"oracle_gumbel_verify failed ({rc})")
    return out


def tv_loss_topk(values, idx, draft, temperature: float = 1.0, grad_scale: float = 1.0, with_grad: bool = True,
                 tie_le: bool = True, clamp_tau=None) -> dict:
    """TV loss against top-K target distributions: values [N, gamma, K]
    (target logits, same storage as draft) at indices idx [N, gamma, K] of
    the vocabulary, renormalised over the K entries; draft [N, gamma, V].
    Returns loss [N], alpha, S, g [N, gamma], flags [N] and grad."""
    v, dt = _logits(values)
    d, dt2 = _logits(draft)
    assert dt == dt2
    N, gamma, V = d.shape
    K = v.shape[-1]
    assert v.shape == (N, gamma, K)
    ix = np.ascontiguousarray(idx, dtype=np.int32).reshape(N, gamma, K)
    out = {"loss": np.empty(N), "alpha": np.empty((N, gamma)), "S": np.empty((N, gamma)),
           "g": np.empty((N, gamma)), "flags": np.empty(N, np.int32)}
    if with_grad:
        out["grad"] = np.empty((N, gamma, V))
    kind, tau = (0, 0.0) if clamp_tau is None else (1, float(clamp_tau))
    rc = _load().oracle_tv_loss_topk(_ptr(v), _ptr(ix), _ptr(d), dt, float(temperature), N, gamma, K, V,
                                     float(grad_scale), int(tie_le), kind, tau, _ptr(out["loss"]), _ptr(out["alpha"]),
                                     _ptr(out["S"]), _ptr(out["g"]), _ptr(out.get("grad")), _ptr(out["flags"]))
    if rc:
        raise RuntimeError(f"oracle_tv_loss_topk failed ({rc})")
    return out


def draft_sample(logits, temperature, uniforms=None, method: str = "multinomial", seed: int = 0,
                 offset: int = 0) -> dict:
    """Draw one token per row of logits [R, V] from softmax(z / T): the
    inverse-CDF draw with uniforms [R] ("multinomial") or the Gumbel-max draw
    with Philox noise ("gumbel", counter (v / 4, 0, r, offset)); T = 0 is
    greedy.  Returns ids [R], flags [R], margin [R]."""
    z, dt = _logits(logits)
    R, V = z.shape
    temp = np.ascontiguousarray(temperature, dtype=np.float64).reshape(R)
    m = {"multinomial": 0, "gumbel": 1}[method]
    u = np.zeros(R) if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float64).reshape(R)
    lo, hi = _seed_words(seed)
    out = {"ids": np.empty(R, np.int32), "flags": np.empty(R, np.int32), "margin": np.empty(R, np.float64)}
    rc = _load().oracle_draft_sample(_ptr(z), dt, _ptr(temp), _ptr(u), m, lo, hi, int(offset) & 0xFFFFFFFF, R, V,
                                     _ptr(out["ids"]), _ptr(out["flags"]), _ptr(out["margin"]))
    if rc:
        raise RuntimeError(f"oracle_draft_sample failed ({rc})")
    return out


def diagnostics(target, draft, temperature) -> dict:
    """Per-position acceptance diagnostics: alpha, tv, ent_q, kl (q || p),
    yhat, p_yhat, rs_better, boundary_margin [B, gamma]; ent_p [B, gamma+1];
    flags [B]."""
    t, dt = _logits(target)
    d, dt2 = _logits(draft)
    assert dt == dt2
    B, g1, V = t.shape
    gamma = g1 - 1
    temp = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    out = {k: np.empty((B, gamma), np.float64) for k in ("alpha", "tv", "ent_q", "kl", "p_yhat", "boundary_margin")}
    out["yhat"] = np.empty((B, gamma), np.int32)
    out["rs_better"] = np.empty((B, gamma), np.int32)
    out["ent_p"] = np.empty((B, gamma + 1), np.float64)
    out["flags"] = np.empty(B, np.int32)
    rc = _load().oracle_diagnostics(_ptr(t), _ptr(d), dt, _ptr(temp), B, gamma, V, _ptr(out["alpha"]), _ptr(out["tv"]),
                                    _ptr(out["ent_q"]), _ptr(out["kl"]), _ptr(out["yhat"]), _ptr(out["p_yhat"]),
                                    _ptr(out["rs_better"]), _ptr(out["boundary_margin"]), _ptr(out["ent_p"]),
                                    _ptr(out["flags"]))
    if rc:
        raise RuntimeError(f"oracle_diagnostics failed ({rc})")
    return out


def row_stats(target, draft, temperature) -> dict:
    """alpha, tv [B, gamma] and entropy [B, gamma+1], flags [B]."""
    t, dt = _logits(target)
    d, _ = _logits(draft)
    B, g1, V = t.shape
    gamma = g1 - 1
    temp = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    out = {"alpha": np.empty((B, gamma)), "tv": np.empty((B, gamma)), "entropy": np.empty((B, g1)),
           "flags": np.empty(B, np.int32)}
    rc = _load().oracle_row_stats(_ptr(t), _ptr(d), dt, _ptr(temp), B, gamma, V, _ptr(out["alpha"]),
                                  _ptr(out["tv"]), _ptr(out["entropy"]), _ptr(out["flags"]))
    if rc:
        raise RuntimeError(f"oracle_row_stats failed ({rc})")
    return out


def tv_loss(target, draft, temperature: float = 1.0, grad_scale: float = 1.0, with_grad: bool = True,
            tie_le: bool = True, shared_target: bool = False, clamp_tau=None) -> dict:
    """TV loss forward/backward over draft [N, gamma, V] and target [N, gamma,
    V] (or, shared_target, [N + gamma - 1, V] with pair (t, k) on row t + k).
    Loss: the e2e loss, or with clamp_tau = tau_max the per-step clamped loss
    sum_k clamp(1 - alpha_k, 0, tau_max).

    Returns loss [N], alpha, S, g [N, gamma] (g = dl/dalpha), flags [N] and
    (with_grad) grad [N, gamma, V] float64.
    """
    t, dt = _logits(target)
    d, _ = _logits(draft)
    N, gamma, V = d.shape
    if shared_target:
        assert t.ndim == 2 and t.shape[0] >= N + gamma - 1 and t.shape[1] == V
    else:
        assert t.shape == d.shape
    out = {"loss": np.empty(N), "alpha": np.empty((N, gamma)), "S": np.empty((N, gamma)),
           "g": np.empty((N, gamma)), "flags": np.empty(N, np.int32)}
    if with_grad:
        out["grad"] = np.empty((N, gamma, V))
    kind, tau = (0, 0.0) if clamp_tau is None else (1, float(clamp_tau))
    rc = _load().oracle_tv_loss_ex(_ptr(t), _ptr(d), dt, float(temperature), N, gamma, V, float(grad_scale),
                                   int(tie_le), int(bool(shared_target)), kind, tau, _ptr(out["loss"]),
                                   _ptr(out["alpha"]), _ptr(out["S"]), _ptr(out["g"]), _ptr(out.get("grad")),
                                   _ptr(out["flags"]))
    if rc:
        raise RuntimeError(f"oracle_tv_loss_ex failed ({rc})")
    return out
