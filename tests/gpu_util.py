"""Helpers shared by the GPU tests: upload host inputs, run the library,
bring outputs back as NumPy arrays."""
import numpy as np
import torch

import mtp_speculative_decoding_row_gb300 as mtp
from mtp_speculative_decoding_row_gb300 import build as mtp_build

DEV = torch.device("cuda:0")


def ensure_library():
    from tests import gpu_util_paths

    if gpu_util_paths.LIBRARY:
        return mtp.load_library(gpu_util_paths.LIBRARY)
    mtp_build.build()
    return mtp.load_library()


def to_dev(a: np.ndarray, dtype: str = None):
    """Host array -> device tensor; uint16 arrays are bfloat16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def to_host_bits(t) -> np.ndarray:
    """Device logits -> host array in the oracle's storage (uint16 for bf16)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


KERNELS = {None: mtp.KERNEL_AUTO, "stream": mtp.KERNEL_STREAM, "resident": mtp.KERNEL_RESIDENT,
           "tmem": mtp.KERNEL_TMEM}


def kcode(name):
    """Kernel choice name (None, "stream", "resident", "tmem") -> mtp_tuning code."""
    return KERNELS[name]


def tune(**fields):
    """Planner overrides through the library's tuning API for a with-block."""
    return mtp.tuning(**fields)


def run_verify(x, with_stats=False):
    out = mtp.mtp_rs_verify(to_dev(x.target), to_dev(x.draft), to_dev(x.draft_ids), to_dev(x.temperature),
                            to_dev(x.uniforms), with_stats=with_stats)
    torch.cuda.synchronize()
    r = {k: (v.cpu().numpy() if v is not None else None) for k, v in out._asdict().items()}
    return r


def run_stats(x):
    out = mtp.mtp_row_stats(to_dev(x.target), to_dev(x.draft), to_dev(x.temperature))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out._asdict().items()}


def run_tv(target, draft, T, scale):
    out = mtp.mtp_tv_loss_fwd_bwd(target, draft, T, scale)
    torch.cuda.synchronize()
    return out
