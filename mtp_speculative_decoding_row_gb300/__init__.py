"""Python binding of the C-ABI library ``libmtprs.so`` (see ``include/mtp_rs.h``).

Argument marshalling only: each function checks the devices, dtypes,
shapes and contiguity of its input tensors and of any caller-supplied
``out`` tensors, allocates missing outputs with PyTorch on the inputs' device,
and calls the C function of the same name on the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and importing a missing library raises.

Method references: "Breaking Entropy Bounds: Accelerating RL Training via MTP
with Rejection Sampling" (§2, §3, §4, §8, App. A, App. F, App. G.1) and
"EntMTP", Related Work "Speculative Decoding".
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

from . import build as _build

__all__ = [
    "mtp_rs_verify", "mtp_to_verify", "mtp_gumbel_verify", "mtp_draft_sample", "mtp_row_stats",
    "mtp_rs_diagnostics", "mtp_tv_loss_fwd_bwd", "mtp_tv_loss_ex", "mtp_tv_loss_topk",
    "mtp_query_plan", "mtp_status_string", "mtp_set_tuning", "mtp_get_tuning", "tuning", "check_row_flags",
    "MTPError", "load_library", "MTP_ERR_TIMEOUT", "KERNEL_AUTO", "KERNEL_STREAM", "KERNEL_RESIDENT", "KERNEL_TMEM",
    "VerifyResult", "TOVerifyResult", "StatsResult", "DiagResult", "TVLossResult", "SampleResult", "ROW_NONFINITE",
    "ROW_BAD_ID", "ROW_BAD_TEMP", "ROW_ZERO_MASS", "ROW_BAD_UNIFORM", "ROW_TIMEOUT", "ERROR_BITS", "MAX_GAMMA", "EXPORTED_SYMBOLS",
]

ROW_NONFINITE, ROW_BAD_ID, ROW_BAD_TEMP, ROW_ZERO_MASS, ROW_BAD_UNIFORM, ROW_TIMEOUT = 1, 2, 4, 8, 16, 32
ERROR_BITS = ROW_NONFINITE | ROW_BAD_ID | ROW_BAD_TEMP | ROW_BAD_UNIFORM | ROW_TIMEOUT
MAX_GAMMA = 32
DTYPE_F32, DTYPE_BF16 = 0, 1
EXPORTED_SYMBOLS = ("mtp_rs_verify", "mtp_to_verify", "mtp_gumbel_verify", "mtp_draft_sample", "mtp_row_stats",
                    "mtp_rs_diagnostics", "mtp_tv_loss_fwd_bwd", "mtp_tv_loss_ex", "mtp_tv_loss_topk",
                    "mtp_query_plan", "mtp_set_tuning", "mtp_get_tuning", "mtp_status_string")
MTP_OK, MTP_ERR_INVALID_ARG, MTP_ERR_UNSUPPORTED_DTYPE, MTP_ERR_MISALIGNED, MTP_ERR_CUDA, MTP_ERR_TIMEOUT, \
    MTP_ERR_NO_DEVICE = range(7)
KERNEL_AUTO, KERNEL_STREAM, KERNEL_RESIDENT, KERNEL_TMEM = range(4)
TUNING_FIELDS = ("cluster_size", "ring_slots", "lookahead", "chunk_vectors", "max_clusters", "verify_kernel",
                 "tv_kernel", "stats_kernel", "tv_resident_drafts", "tv_l2_mb", "pair_l2_mb", "row_streams",
                 "fault_wait_us", "fault_skip_position")


class _Tuning(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in TUNING_FIELDS]


PLAN_OPS = {"verify": 0, "verify_stats": 1, "row_stats": 2, "tv_loss": 3, "verify_resident": 4,
            "tv_loss_resident": 5, "diagnostics": 6, "row_stats_resident": 7, "to_verify": 8, "gumbel_verify": 9,
            "draft_sample": 10, "draft_sample_gumbel": 11}

_lib = None


class MTPError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {mtp_status_string(status)} (status {status})")
        self.status = status


def load_library(path: Optional[str] = None, build_if_missing: bool = False):
    """Load libmtprs.so (ctypes) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        if build_if_missing:
            _build.build()
        else:
            raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
                              f"g.build()'` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.mtp_rs_verify.argtypes = [P, P, I, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.mtp_rs_verify.restype = I
    lib.mtp_to_verify.argtypes = [P, P, I, P, P, I, I, I, P, P, P, P, P]
    lib.mtp_to_verify.restype = I
    lib.mtp_row_stats.argtypes = [P, P, I, P, I, I, I, P, P, P, P]
    lib.mtp_row_stats.restype = I
    lib.mtp_draft_sample.argtypes = [P, I, P, P, I, ctypes.c_uint64, ctypes.c_uint32, I, I, P, P, P]
    lib.mtp_draft_sample.restype = I
    lib.mtp_tv_loss_topk.argtypes = [P, P, P, I, F, I, I, I, I, F, I, F, P, P, P, P, P]
    lib.mtp_tv_loss_topk.restype = I
    lib.mtp_tv_loss_ex.argtypes = [P, P, I, F, I, I, I, F, I, I, F, P, P, P, P, P]
    lib.mtp_tv_loss_ex.restype = I
    lib.mtp_gumbel_verify.argtypes = [P, P, I, P, P, P, ctypes.c_uint64, ctypes.c_uint32, I, I, I, P, P, P, P]
    lib.mtp_gumbel_verify.restype = I
    lib.mtp_rs_diagnostics.argtypes = [P, P, I, P, I, I, I, P, P, P, P, P, P, P, P, P]
    lib.mtp_rs_diagnostics.restype = I
    lib.mtp_tv_loss_fwd_bwd.argtypes = [P, P, I, F, I, I, I, F, P, P, P, P, P]
    lib.mtp_tv_loss_fwd_bwd.restype = I
    lib.mtp_query_plan.argtypes = [I, I, I, I, I, P, P, P, P]
    lib.mtp_query_plan.restype = I
    lib.mtp_set_tuning.argtypes = [P]
    lib.mtp_set_tuning.restype = I
    lib.mtp_get_tuning.argtypes = [P]
    lib.mtp_get_tuning.restype = I
    lib.mtp_status_string.argtypes = [I]
    lib.mtp_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def mtp_query_plan(op: str, dtype: str, units: int, gamma: int, V: int) -> dict:
    """Launch plan of a call on the current device: cluster size, persistent
    clusters, shared memory per CTA and ``resident_drafts`` (cluster-resident
    TV kernel: draft slices kept on chip, 0 for the streaming TV kernel;
    "verify": ring slots per warp of the streaming kernel, 0 when the call
    would use the cluster-resident kernel)."""
    vals = [ctypes.c_int(0) for _ in range(4)]
    rc = load_library().mtp_query_plan(PLAN_OPS[op], DTYPE_BF16 if dtype == "bf16" else DTYPE_F32, units, gamma, V,
                                       *[ctypes.byref(v) for v in vals])
    if rc:
        raise MTPError("mtp_query_plan", rc)
    return dict(zip(("cluster_size", "clusters", "smem_bytes", "resident_drafts"), (v.value for v in vals)))


def mtp_status_string(status: int) -> str:
    return load_library().mtp_status_string(int(status)).decode()


def mtp_set_tuning(**fields) -> None:
    """Set the process-wide planner overrides (see mtp_tuning in
    include/mtp_rs.h); no argument clears them.  Field names: TUNING_FIELDS;
    a value of 0 or None keeps the planner's choice for that field."""
    unknown = set(fields) - set(TUNING_FIELDS)
    if unknown:
        raise ValueError(f"unknown tuning fields {sorted(unknown)}")
    t = _Tuning(*(int(fields.get(name) or 0) for name in TUNING_FIELDS))
    rc = load_library().mtp_set_tuning(ctypes.byref(t))
    if rc:
        raise MTPError("mtp_set_tuning", rc)


def mtp_get_tuning() -> dict:
    t = _Tuning()
    rc = load_library().mtp_get_tuning(ctypes.byref(t))
    if rc:
        raise MTPError("mtp_get_tuning", rc)
    return {name: getattr(t, name) for name in TUNING_FIELDS}


class tuning:
    """Context manager: planner overrides for the calls made inside it, the
    previous overrides restored on exit (``with tuning(cluster_size=8): ...``).
    Fields given as None keep the planner's choice."""

    def __init__(self, **fields):
        self.fields = fields

    def __enter__(self):
        self.old = mtp_get_tuning()
        new = dict(self.old)
        new.update({k: (v or 0) for k, v in self.fields.items()})
        mtp_set_tuning(**new)
        return self

    def __exit__(self, *exc):
        mtp_set_tuning(**self.old)
        return False


def check_row_flags(row_flags) -> None:
    """Raise MTPError(MTP_ERR_TIMEOUT) if any row of a finished call carries
    ROW_TIMEOUT (an on-chip wait gave up).  Synchronises with the tensor's
    stream by reading it back."""
    flags = row_flags.cpu() if hasattr(row_flags, "cpu") else row_flags
    if bool(((flags & ROW_TIMEOUT) != 0).any()):
        raise MTPError("device", MTP_ERR_TIMEOUT)


# ------------------------------------------------------------ marshalling --

def _torch():
    import torch

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _check(t, name, device, dtype=None, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and (not t.is_cuda or t.device != device):
        raise ValueError(f"{name} must be a CUDA tensor on {device}")


def _check_out(out, specs, device, fn: str):
    """Check every field of a caller-supplied result tuple: (name, dtype,
    shape, required).  A missing required field, or a field of another
    device, dtype or shape, or non-contiguous, raises before any launch."""
    given = []
    for name, dtype, shape, required in specs:
        t = getattr(out, name)
        if t is None:
            if required:
                raise ValueError(f"{fn}: out.{name} is required")
            continue
        _check(t, f"out.{name}", None, dtype, shape)
        given.append((t, name))
    for t, name in given:
        _check(t, f"out.{name}", device)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device, stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


class VerifyResult(NamedTuple):
    tokens: "object"      # [B, gamma+1] int32, -1 padded
    accept_len: "object"  # [B] int32 (-1 if flagged)
    alpha: "object"       # [B, gamma] float32 or None
    entropy: "object"     # [B, gamma+1] float32 or None
    row_flags: "object"   # [B] int32


class TOVerifyResult(NamedTuple):
    tokens: "object"        # [B, gamma+1] int32, -1 padded
    accept_len: "object"    # [B] int32 (-1 if flagged)
    draft_tokens: "object"  # [B, gamma] int32: arg max draft token of each decided position, -1 elsewhere
    row_flags: "object"     # [B] int32


class StatsResult(NamedTuple):
    alpha: "object"
    entropy: "object"
    row_flags: "object"


class DiagResult(NamedTuple):
    alpha: "object"      # [B, gamma] float32: sum min(p, q) = 1 - d_TV
    ent_p: "object"      # [B, gamma+1] float32: H(p) in nats
    ent_q: "object"      # [B, gamma] float32: H(q) in nats
    kl: "object"         # [B, gamma] float32: D_KL(q || p) in nats
    yhat: "object"       # [B, gamma] int32: arg max of the draft logits
    p_yhat: "object"     # [B, gamma] float32: p(yhat)
    rs_better: "object"  # [B, gamma] int32: 1 if d_TV < 1 - p(yhat)
    row_flags: "object"  # [B] int32


class TVLossResult(NamedTuple):
    loss: "object"        # [N] float32
    alpha: "object"       # [N, gamma] float32
    grad: "object"        # [N, gamma, V] float32
    row_flags: "object"   # [N] int32


def mtp_rs_verify(target_logits, draft_logits, draft_ids, temperature, uniforms, *, with_stats: bool = False,
                  out: Optional[VerifyResult] = None, stream=None) -> VerifyResult:
    """Batched MTP rejection-sampling verification (see mtp_rs_verify in
    include/mtp_rs.h).  target_logits [B, gamma+1, V], draft_logits
    [B, gamma, V] (float32 or bfloat16), draft_ids [B, gamma] int32,
    temperature [B] float32, uniforms [B, gamma+1] float32."""
    torch = _torch()
    dev = target_logits.device
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if out is not None:
        if (out.alpha is None) != (out.entropy is None) or (out.alpha is not None) != bool(with_stats):
            raise ValueError("mtp_rs_verify: out.alpha and out.entropy must both be given iff with_stats")
        _check_out(out, [("tokens", torch.int32, (B, gamma + 1), True), ("accept_len", torch.int32, (B,), True),
                         ("alpha", torch.float32, (B, gamma), False), ("entropy", torch.float32, (B, gamma + 1), False),
                         ("row_flags", torch.int32, (B,), False)], dev, "mtp_rs_verify")
    _check(target_logits, "target_logits", dev)
    _check(draft_logits, "draft_logits", dev, target_logits.dtype, (B, gamma, V))
    _check(draft_ids, "draft_ids", dev, torch.int32, (B, gamma))
    _check(temperature, "temperature", dev, torch.float32, (B,))
    _check(uniforms, "uniforms", dev, torch.float32, (B, gamma + 1))
    if out is None:
        out = VerifyResult(
            torch.empty((B, gamma + 1), dtype=torch.int32, device=dev),
            torch.empty((B,), dtype=torch.int32, device=dev),
            torch.empty((B, gamma), dtype=torch.float32, device=dev) if with_stats else None,
            torch.empty((B, gamma + 1), dtype=torch.float32, device=dev) if with_stats else None,
            torch.empty((B,), dtype=torch.int32, device=dev))
    rc = load_library().mtp_rs_verify(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_ids), _ptr(temperature),
        _ptr(uniforms), B, gamma, V, _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.alpha), _ptr(out.entropy),
        _ptr(out.row_flags), _stream(dev, stream))
    if rc:
        raise MTPError("mtp_rs_verify", rc)
    return out


def mtp_to_verify(target_logits, draft_logits, temperature, uniforms, *, out: Optional["TOVerifyResult"] = None,
                  stream=None) -> "TOVerifyResult":
    """Batched target-only verification (see mtp_to_verify in
    include/mtp_rs.h): the draft token of each position is the arg max of its
    draft logits, accepted iff u < p(y).  Returns tokens [B, gamma+1],
    accept_len [B], draft_tokens [B, gamma] and row_flags [B]."""
    torch = _torch()
    dev = target_logits.device
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if out is not None:
        _check_out(out, [("tokens", torch.int32, (B, gamma + 1), True), ("accept_len", torch.int32, (B,), True),
                         ("draft_tokens", torch.int32, (B, gamma), False), ("row_flags", torch.int32, (B,), False)],
                   dev, "mtp_to_verify")
    _check(target_logits, "target_logits", dev)
    _check(draft_logits, "draft_logits", dev, target_logits.dtype, (B, gamma, V))
    _check(temperature, "temperature", dev, torch.float32, (B,))
    _check(uniforms, "uniforms", dev, torch.float32, (B, gamma + 1))
    if out is None:
        out = TOVerifyResult(
            torch.empty((B, gamma + 1), dtype=torch.int32, device=dev),
            torch.empty((B,), dtype=torch.int32, device=dev),
            torch.empty((B, gamma), dtype=torch.int32, device=dev),
            torch.empty((B,), dtype=torch.int32, device=dev))
    rc = load_library().mtp_to_verify(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(temperature), _ptr(uniforms), B,
        gamma, V, _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.draft_tokens), _ptr(out.row_flags),
        _stream(dev, stream))
    if rc:
        raise MTPError("mtp_to_verify", rc)
    return out


def mtp_gumbel_verify(target_logits, draft_logits, draft_ids, temperature, uniforms, seed: int, offset: int = 0, *,
                      out: Optional[VerifyResult] = None, stream=None) -> VerifyResult:
    """Rejection-sampling verification whose final token (residual or bonus)
    is a Gumbel-max draw with in-kernel Philox noise keyed by (seed, offset,
    sequence, row); u[:, gamma] is not read.  Returns tokens, accept_len and
    row_flags (alpha and entropy None)."""
    torch = _torch()
    dev = target_logits.device
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if out is not None:
        if out.alpha is not None or out.entropy is not None:
            raise ValueError("mtp_gumbel_verify: out.alpha and out.entropy must be None")
        _check_out(out, [("tokens", torch.int32, (B, g1), True), ("accept_len", torch.int32, (B,), True),
                         ("row_flags", torch.int32, (B,), False)], dev, "mtp_gumbel_verify")
    _check(target_logits, "target_logits", dev)
    _check(draft_logits, "draft_logits", dev, target_logits.dtype, (B, gamma, V))
    _check(draft_ids, "draft_ids", dev, torch.int32, (B, gamma))
    _check(temperature, "temperature", dev, torch.float32, (B,))
    _check(uniforms, "uniforms", dev, torch.float32, (B, g1))
    if out is None:
        out = VerifyResult(torch.empty((B, g1), dtype=torch.int32, device=dev),
                           torch.empty((B,), dtype=torch.int32, device=dev), None, None,
                           torch.empty((B,), dtype=torch.int32, device=dev))
    rc = load_library().mtp_gumbel_verify(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_ids), _ptr(temperature),
        _ptr(uniforms), int(seed) & ((1 << 64) - 1), int(offset) & 0xFFFFFFFF, B, gamma, V, _ptr(out.tokens),
        _ptr(out.accept_len), _ptr(out.row_flags), _stream(dev, stream))
    if rc:
        raise MTPError("mtp_gumbel_verify", rc)
    return out


class SampleResult(NamedTuple):
    ids: "object"        # [R] int32 (-1 for a flagged row)
    row_flags: "object"  # [R] int32


def mtp_draft_sample(draft_logits, temperature, uniforms=None, *, method: str = "multinomial", seed: int = 0,
                     offset: int = 0, out: Optional[SampleResult] = None, stream=None) -> SampleResult:
    """One draft token per row of logits [..., V] (flattened to [R, V]) from
    softmax(z / T): inverse CDF with uniforms [R] ("multinomial") or the
    Gumbel-max draw with in-kernel Philox noise ("gumbel"); T = 0 is greedy."""
    torch = _torch()
    dev = draft_logits.device
    V = draft_logits.shape[-1]
    R = draft_logits.numel() // V if V else 0
    if out is not None:
        _check_out(out, [("ids", torch.int32, (R,), True), ("row_flags", torch.int32, (R,), False)], dev,
                   "mtp_draft_sample")
    _check(draft_logits, "draft_logits", dev)
    _check(temperature, "temperature", dev, torch.float32)
    if temperature.numel() != R:
        raise ValueError(f"temperature must have {R} entries")
    m = {"multinomial": 0, "gumbel": 1}[method]
    if m == 0:
        if uniforms is None:
            raise ValueError("the multinomial draw needs uniforms")
        _check(uniforms, "uniforms", dev, torch.float32)
        if uniforms.numel() != R:
            raise ValueError(f"uniforms must have {R} entries")
    if out is None:
        out = SampleResult(torch.empty((R,), dtype=torch.int32, device=dev),
                           torch.empty((R,), dtype=torch.int32, device=dev))
    rc = load_library().mtp_draft_sample(
        _ptr(draft_logits), _dtype_code(draft_logits), _ptr(temperature), _ptr(uniforms) if m == 0 else None, m,
        int(seed) & ((1 << 64) - 1), int(offset) & 0xFFFFFFFF, R, V, _ptr(out.ids), _ptr(out.row_flags),
        _stream(dev, stream))
    if rc:
        raise MTPError("mtp_draft_sample", rc)
    return out


def mtp_row_stats(target_logits, draft_logits, temperature, *, out: Optional[StatsResult] = None,
                  stream=None) -> StatsResult:
    """Per-position alpha = sum min(p, q) [B, gamma] and H(p) [B, gamma+1]."""
    torch = _torch()
    dev = target_logits.device
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if out is not None:
        _check_out(out, [("alpha", torch.float32, (B, gamma), True), ("entropy", torch.float32, (B, g1), True),
                         ("row_flags", torch.int32, (B,), False)], dev, "mtp_row_stats")
    _check(target_logits, "target_logits", dev)
    _check(draft_logits, "draft_logits", dev, target_logits.dtype, (B, gamma, V))
    _check(temperature, "temperature", dev, torch.float32, (B,))
    if out is None:
        out = StatsResult(torch.empty((B, gamma), dtype=torch.float32, device=dev),
                          torch.empty((B, g1), dtype=torch.float32, device=dev),
                          torch.empty((B,), dtype=torch.int32, device=dev))
    rc = load_library().mtp_row_stats(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(temperature), B, gamma, V,
        _ptr(out.alpha), _ptr(out.entropy), _ptr(out.row_flags), _stream(dev, stream))
    if rc:
        raise MTPError("mtp_row_stats", rc)
    return out


def mtp_rs_diagnostics(target_logits, draft_logits, temperature, *, out: Optional[DiagResult] = None,
                       stream=None) -> DiagResult:
    """Per-position acceptance diagnostics (no decisions): alpha, H(p), H(q),
    D_KL(q || p), the arg max draft token, its target probability and the
    rejection-sampling-better test d_TV < 1 - p(yhat)."""
    torch = _torch()
    dev = target_logits.device
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if out is not None:
        f32, i32 = torch.float32, torch.int32
        _check_out(out, [("alpha", f32, (B, gamma), False), ("ent_p", f32, (B, g1), False),
                         ("ent_q", f32, (B, gamma), False), ("kl", f32, (B, gamma), False),
                         ("yhat", i32, (B, gamma), False), ("p_yhat", f32, (B, gamma), False),
                         ("rs_better", i32, (B, gamma), False), ("row_flags", i32, (B,), False)], dev,
                   "mtp_rs_diagnostics")
    _check(target_logits, "target_logits", dev)
    _check(draft_logits, "draft_logits", dev, target_logits.dtype, (B, gamma, V))
    _check(temperature, "temperature", dev, torch.float32, (B,))
    if out is None:
        f = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)  # noqa: E731
        i = lambda *shape: torch.empty(shape, dtype=torch.int32, device=dev)  # noqa: E731
        out = DiagResult(f(B, gamma), f(B, g1), f(B, gamma), f(B, gamma), i(B, gamma), f(B, gamma), i(B, gamma),
                         i(B))
    rc = load_library().mtp_rs_diagnostics(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(temperature), B, gamma, V,
        _ptr(out.alpha), _ptr(out.ent_p), _ptr(out.ent_q), _ptr(out.kl), _ptr(out.yhat), _ptr(out.p_yhat),
        _ptr(out.rs_better), _ptr(out.row_flags), _stream(dev, stream))
    if rc:
        raise MTPError("mtp_rs_diagnostics", rc)
    return out


def mtp_tv_loss_topk(target_values, target_idx, draft_logits, temperature: float = 1.0, grad_scale: float = 1.0, *,
                     clamp_tau: Optional[float] = None, out: Optional[TVLossResult] = None,
                     stream=None) -> TVLossResult:
    """Fused TV loss forward + backward against top-K targets: values and
    int32 indices [N, gamma, K] of the target's K cached logits (softmax
    renormalised over them), draft logits [N, gamma, V]."""
    torch = _torch()
    dev = draft_logits.device
    N, gamma, V = draft_logits.shape
    K = target_values.shape[-1]
    if out is not None:
        _check_out(out, [("loss", torch.float32, (N,), True), ("alpha", torch.float32, (N, gamma), False),
                         ("grad", torch.float32, (N, gamma, V), True), ("row_flags", torch.int32, (N,), False)], dev,
                   "mtp_tv_loss_topk")
    _check(draft_logits, "draft_logits", dev)
    _check(target_values, "target_values", dev, draft_logits.dtype, (N, gamma, K))
    _check(target_idx, "target_idx", dev, torch.int32, (N, gamma, K))
    if out is None:
        out = TVLossResult(torch.empty((N,), dtype=torch.float32, device=dev),
                           torch.empty((N, gamma), dtype=torch.float32, device=dev),
                           torch.empty((N, gamma, V), dtype=torch.float32, device=dev),
                           torch.empty((N,), dtype=torch.int32, device=dev))
    rc = load_library().mtp_tv_loss_topk(
        _ptr(target_values), _ptr(target_idx), _ptr(draft_logits), _dtype_code(draft_logits), float(temperature), N,
        gamma, K, V, float(grad_scale), 0 if clamp_tau is None else 1, 0.0 if clamp_tau is None else float(clamp_tau),
        _ptr(out.loss), _ptr(out.alpha), _ptr(out.grad), _ptr(out.row_flags), _stream(dev, stream))
    if rc:
        raise MTPError("mtp_tv_loss_topk", rc)
    return out


def mtp_tv_loss_fwd_bwd(target_logits, draft_logits, temperature: float = 1.0, grad_scale: float = 1.0, *,
                        shared_target: bool = False, clamp_tau: Optional[float] = None,
                        out: Optional[TVLossResult] = None, stream=None) -> TVLossResult:
    """Fused TV loss forward + backward over draft logits [N, gamma, V];
    returns per-position loss, alpha, the float32 gradient w.r.t. the draft
    logits and row flags.  Target logits are [N, gamma, V], or with
    shared_target [N + gamma - 1, V] (pair (t, k) on row t + k).  The loss is
    the e2e loss, or with clamp_tau = tau_max the per-step clamped loss
    sum_k clamp(1 - alpha_k, 0, tau_max)."""
    torch = _torch()
    dev = draft_logits.device
    N, gamma, V = draft_logits.shape
    if out is not None:
        _check_out(out, [("loss", torch.float32, (N,), True), ("alpha", torch.float32, (N, gamma), False),
                         ("grad", torch.float32, (N, gamma, V), True), ("row_flags", torch.int32, (N,), False)], dev,
                   "mtp_tv_loss_fwd_bwd")
    _check(draft_logits, "draft_logits", dev)
    if shared_target:
        if target_logits.dim() != 2 or target_logits.shape[0] < N + gamma - 1 or target_logits.shape[1] != V:
            raise ValueError(f"shared target_logits must be [>= N + gamma - 1, V], got {tuple(target_logits.shape)}")
        _check(target_logits, "target_logits", dev, draft_logits.dtype)
    else:
        _check(target_logits, "target_logits", dev, draft_logits.dtype, (N, gamma, V))
    if out is None:
        out = TVLossResult(torch.empty((N,), dtype=torch.float32, device=dev),
                           torch.empty((N, gamma), dtype=torch.float32, device=dev),
                           torch.empty((N, gamma, V), dtype=torch.float32, device=dev),
                           torch.empty((N,), dtype=torch.int32, device=dev))
    lib = load_library()
    if not shared_target and clamp_tau is None:
        rc = lib.mtp_tv_loss_fwd_bwd(
            _ptr(target_logits), _ptr(draft_logits), _dtype_code(draft_logits), float(temperature), N, gamma, V,
            float(grad_scale), _ptr(out.loss), _ptr(out.alpha), _ptr(out.grad), _ptr(out.row_flags),
            _stream(dev, stream))
        name = "mtp_tv_loss_fwd_bwd"
    else:
        rc = lib.mtp_tv_loss_ex(
            _ptr(target_logits), _ptr(draft_logits), _dtype_code(draft_logits), float(temperature), N, gamma, V,
            float(grad_scale), int(bool(shared_target)), 0 if clamp_tau is None else 1,
            0.0 if clamp_tau is None else float(clamp_tau), _ptr(out.loss), _ptr(out.alpha), _ptr(out.grad),
            _ptr(out.row_flags), _stream(dev, stream))
        name = "mtp_tv_loss_ex"
    if rc:
        raise MTPError(name, rc)
    return out
