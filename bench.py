"""Benchmark: verified draft positions per second and logit GB/s (fraction of
the measured HBM roofline) at V = 151,936 on one GB300.

Step = one call of the hot path over one batch of synthetic input.  The
headline workload is the RL-rollout verify batch (B = 512 sequences,
gamma = 3, V = 151,936, bf16 logits; peaked Zipf(1.1)+8 rows with 30 %
N(0, 1) rows, delta in {0.1, 0.5}, T in {0.6, 1.0}): one mtp_rs_verify call
per step.  The same JSON line also reports the other workloads measured in
the same run: the B = 64 verify batch, deep speculation with per-position
alpha and entropy (B = 256, gamma = 7, fp32), row statistics, diagnostics,
the acceptance-method variants, draft sampling and the e2e TV-loss
forward+backward (N = 16,384) with its variants.

Timing: inputs resident in HBM; several copies of each input are rotated so
successive steps never hit L2 (each copy is > L2 or the rotation exceeds 4x
L2); steps are replayed from a captured CUDA graph and timed with CUDA events
on the launching stream, synchronised on both sides.  `e2e` measures the same
metric through the public API with pinned host buffers: host-to-device copy
of the step's inputs, the call, and the device-to-host copy of its outputs.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {cuda,reference}]
       [--workloads rl512,verify64,deep256,stats256,diag256,to64,gumbel64,sample192,gsample192,tvloss,
                    tvshared,tvtopk] [--cpu-baselines {all,headline,none}]
Under torchrun each rank runs its own replica (weak scaling); rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and logit GB/s (% of HBM roofline) at V=151936"
UNIT = "positions/s"
L2_BYTES = 129 * 1024 * 1024

# Source files of each kernel family (the kernel and the headers it uses).
KERNEL_FILES = {
    "stream": ["stream_kernels.cu", "chunk_math.cuh", "common.cuh", "philox.cuh", "kernels.h", "gsample.h"],
    "tv_tmem": ["tv_tmem_kernels.cu", "chunk_math.cuh", "common.cuh", "tmem.cuh", "kernels.h"],
    "row": ["row_kernels.cu", "common.cuh", "kernels.h"],
    "pair": ["pair_stream_kernels.cu", "chunk_math.cuh", "common.cuh", "kernels.h"],
    "tv_stream": ["tv_stream_kernels.cu", "chunk_math.cuh", "common.cuh", "kernels.h"],
}

# dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed
# ncu captures (profiles/), keyed by workload: valid only while the kernel's
# source files hash to the value they were captured on (null otherwise).
# Captures on a reduced case are scaled to the workload by the units
# processed (traffic grows in proportion; profiles/ says which).
TRAFFIC = {
    # stream_kernel_impl<bf16_t,160,0>, rl512 in full: 1,066,138,368 read + 3,778,560 written
    # (profiles/stream_kernel_rl512.md)
    "rl512": {"bytes": 1069916928, "family": "stream", "csrc": "5e20b20ae3cf8a29"},
    # stream_kernel_impl<bf16_t,128,2> (Gumbel-max verify) in full: 132,694,016 + 6,277,376 bytes
    # (profiles/stream_kernel_gumbel64.md)
    "gumbel64": {"bytes": 138971392, "family": "stream", "csrc": "5e20b20ae3cf8a29"},
    # gsample_kernel_impl<bf16_t> (Gumbel-max draft sampling, one pass) in full: 63,138,816 +
    # 500,480 bytes (profiles/gsample_kernel_gsample192.md)
    "gsample192": {"bytes": 63639296, "family": "stream", "csrc": "5e20b20ae3cf8a29"},
    # tvm_kernel_impl<bf16_t,10> at N = 512 (1,123,948,800 read + 872,851,968 written) x 32
    # for N = 16,384 (profiles/tv_tmem_kernel_tvloss_n512.md)
    "tvloss": {"bytes": 63897624576, "family": "tv_tmem", "csrc": "04c6799a1030e40f"},
    # tvs_kernel_impl<bf16_t,160,1> (top-K targets) at N = 512 (691,457,280 read + 873,746,176
    # written) x 32 for N = 16,384, the same launch plan (profiles/tv_stream_kernel_tvtopk_n512.md)
    "tvtopk": {"bytes": 50086510592, "family": "tv_stream", "csrc": "f7118740f92f9310"},
    # row_kernel_impl<float,2> (statistics) and <float,1> (verify with statistics) on the first 64
    # sequences of deep256 (583,515,392 + 3,678,976 and 583,566,080 + 3,705,088 bytes) x 4 for
    # B = 256 (profiles/row_kernel_deep256_b64.md)
    "stats256": {"bytes": 2348777472, "family": "row", "csrc": "903c4eee388664e8"},
    "deep256": {"bytes": 2349084672, "family": "row", "csrc": "903c4eee388664e8"},
}


def csrc_hash(family: str = None) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mtp_speculative_decoding_row_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(csrc, "*"))) if family is None else \
        [os.path.join(csrc, f) for f in KERNEL_FILES[family]]
    for p in files:
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(name: str):
    """ncu DRAM bytes per launch of the workload, or None when the capture is
    missing or its kernel sources have changed since."""
    tr = TRAFFIC.get(name)
    if not tr or tr.get("csrc") != csrc_hash(tr["family"]):
        return None
    return tr["bytes"]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------ distributed --

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "cuda" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def max_over_ranks(pg, x: float, device=None) -> float:
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except FileNotFoundError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.rows.append(parts)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = self.rows
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# -------------------------------------------------------------- workloads --

def alg_bytes_verify(accept_len: np.ndarray, gamma: int, V: int, es: int, stats: bool) -> int:
    """Logit bytes the method must read.  Without statistics the verify
    stops at the first rejection: (n+1) target rows and min(n+1, gamma)
    draft rows per sequence; with statistics every row is read."""
    B = accept_len.shape[0]
    if stats:
        return B * (2 * gamma + 1) * V * es
    n = accept_len.astype(np.int64)
    return int(((n + 1) + np.minimum(n + 1, gamma)).sum()) * V * es


TV_WORKLOADS = ("tvloss", "tvshared", "tvtopk")

# Host input sets drawn so far, by configuration name.
_INPUTS = {}

# Workloads that run another call on the inputs of a named configuration:
# (input config, call).
STATS_WORKLOADS = {"stats256": ("deep256", "stats"), "diag256": ("deep256", "diag"),
                   "to64": ("verify64", "to"), "gumbel64": ("verify64", "gumbel"),
                   "sample192": ("verify64", "sample"), "gsample192": ("verify64", "gsample")}


class VerifyWorkload:
    def __init__(self, name: str, device, copies: int, deep_b=None):
        import torch

        import workloads as W
        import mtp_speculative_decoding_row_gb300 as mtp

        self.mtp = mtp
        base_name, self.kind = STATS_WORKLOADS.get(name, (name, "verify"))
        if base_name not in _INPUTS:  # several workloads share one input set: draw it once
            _INPUTS[base_name] = W.config(base_name)
        self.x = x = _INPUTS[base_name]
        if deep_b and base_name == "deep256" and deep_b < x.B:
            x = W.subset(x, deep_b)  # the first deep_b sequences (profiling cases)
            self.x = x
        self.name, self.device = name, device
        self.B, self.gamma, self.V, self.es = x.B, x.gamma, x.V, x.esize
        self.stats = x.want_stats or self.kind in ("stats", "diag")
        self.sample_args = None

        def up(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
            return torch.from_numpy(a).to(device)

        base = [up(x.target), up(x.draft), up(x.draft_ids), up(x.temperature), up(x.uniforms)]
        self.inputs = [base] + [[t.clone() for t in base] for _ in range(copies - 1)]
        self.copies = copies
        self.outs = [None] * copies
        self.positions = x.B * x.gamma
        self.bytes_full = x.B * (2 * x.gamma + 1) * x.V * x.esize

    def call(self, i: int, stream=None):
        t, d, ids, T, u = self.inputs[i % self.copies]
        o = self.outs[i % self.copies]
        if self.kind == "stats":
            o = self.mtp.mtp_row_stats(t, d, T, out=o, stream=stream)
        elif self.kind == "diag":
            o = self.mtp.mtp_rs_diagnostics(t, d, T, out=o, stream=stream)
        elif self.kind == "to":
            o = self.mtp.mtp_to_verify(t, d, T, u, out=o, stream=stream)
        elif self.kind == "gumbel":
            o = self.mtp.mtp_gumbel_verify(t, d, ids, T, u, 1234, i % self.copies, out=o, stream=stream)
        elif self.kind in ("sample", "gsample"):
            if self.sample_args is None:
                self.sample_args = [None] * self.copies
            if self.sample_args[i % self.copies] is None:
                # per row: the sequence's temperature and one uniform per draft step
                self.sample_args[i % self.copies] = (T.repeat_interleave(self.gamma).contiguous(),
                                                     u[:, :self.gamma].reshape(-1).contiguous())
            Tr, ur = self.sample_args[i % self.copies]
            o = self.mtp.mtp_draft_sample(d, Tr, ur, method="multinomial" if self.kind == "sample" else "gumbel",
                                          seed=4321, offset=i % self.copies, out=o, stream=stream)
        else:
            o = self.mtp.mtp_rs_verify(t, d, ids, T, u, with_stats=self.stats, out=o, stream=stream)
        self.outs[i % self.copies] = o

    def alg_bytes(self) -> int:
        if self.kind in ("stats", "diag"):
            return self.bytes_full
        if self.kind in ("sample", "gsample"):
            return self.B * self.gamma * self.V * self.es  # every draft row once
        n = self.outs[0].accept_len.cpu().numpy()
        return alg_bytes_verify(n, self.gamma, self.V, self.es, self.stats)

    def plan_op(self) -> str:
        return {"stats": "row_stats", "diag": "diagnostics", "to": "to_verify", "gumbel": "gumbel_verify",
                "sample": "draft_sample", "gsample": "draft_sample_gumbel"}.get(
            self.kind, "verify_stats" if self.stats else "verify")

    def describe(self) -> str:
        x = self.x
        return {"verify64": "verify batch: B=64 gamma=3 V=151936 bf16 logits, entropy-spanning target (0.5-4 nats), "
                            "draft = target + N(0,0.3), draft ids ~ q, T=1",
                "rl512": "RL rollout verify: B=512 gamma=3 V=151936 bf16, peaked Zipf(1.1)+8 rows, 30% N(0,1) rows, "
                         "delta in {0.1,0.5}, T in {0.6,1.0}",
                "deep256": "deep speculation + stats: B=256 gamma=7 V=151936 fp32, T in {0.6,0.8,1.0}, delta 0..1, "
                           "alpha and H for every position",
                "stats256": "row statistics (alpha, H(p)) without decisions on the deep256 inputs: B=256 gamma=7 "
                            "V=151936 fp32",
                "diag256": "acceptance diagnostics (alpha, H(p), H(q), KL(q||p), arg max draft, p(yhat), "
                           "rs_better) on the deep256 inputs: B=256 gamma=7 V=151936 fp32",
                "to64": "target-only verification (arg max drafts, accept iff u < p(yhat)) on the verify64 inputs",
                "gumbel64": "rejection sampling with the Gumbel-max final draw (in-kernel Philox noise) on the "
                            "verify64 inputs",
                "sample192": "draft sampling by inverse CDF: the 192 draft rows (64 x 3) of verify64, V=151936 bf16",
                "gsample192": "draft sampling by Gumbel-max (in-kernel Philox noise): the 192 draft rows of verify64"
                }[self.name]


class TVWorkload:
    TOPK = 64  # cached target entries per pair in the top-K workload

    def __init__(self, device, N=None, shared=False, topk=False):
        import torch

        import workloads as W
        import mtp_speculative_decoding_row_gb300 as mtp

        self.mtp = mtp
        self.shared = shared
        self.topk = topk
        if shared:
            N = N or 16384
            self.x = x = W.tvloss_shared_inputs_device("tvshared", N, 3, W.V_QWEN, W.CONFIG_NAMES.index("tvloss"),
                                                       device)
        else:
            self.x = x = W.config("tvloss", device=device, N_override=N)
        self.N, self.gamma, self.V, self.es = x.N, x.gamma, x.V, 2
        self.stats = False
        self.out = None
        self.copies = 1
        self.positions = x.N * x.gamma
        if topk:
            # the target cached as its K largest logits per pair (input preparation, not timed)
            vals, idx = torch.topk(x.target, self.TOPK, dim=-1)
            self.tk_vals, self.tk_idx = vals.contiguous(), idx.to(torch.int32).contiguous()
            x.target = None
            torch.cuda.empty_cache()
        # draft read (2 B) and gradient written (4 B) per (t, k, v); target rows read once
        if topk:
            tgt = x.N * x.gamma * self.TOPK * (2 + 4)
        else:
            tgt = (x.N + x.gamma - 1) * x.V * 2 if shared else x.N * x.gamma * x.V * 2
        self.bytes_full = x.N * x.gamma * x.V * (2 + 4) + tgt

    def call(self, i: int, stream=None):
        if self.topk:
            self.out = self.mtp.mtp_tv_loss_topk(self.tk_vals, self.tk_idx, self.x.draft, self.x.temperature,
                                                 self.x.grad_scale, out=self.out, stream=stream)
            return
        self.out = self.mtp.mtp_tv_loss_fwd_bwd(self.x.target, self.x.draft, self.x.temperature, self.x.grad_scale,
                                                shared_target=self.shared, out=self.out, stream=stream)

    def alg_bytes(self) -> int:
        return self.bytes_full

    def describe(self) -> str:
        if self.topk:
            return (f"e2e TV loss fwd+bwd against top-K targets (K={self.TOPK} cached target logits per pair, "
                    f"renormalised): N={self.N} positions x gamma=3, V=151936, bf16, fp32 gradient, T=1")
        if self.shared:
            return (f"e2e TV loss fwd+bwd, shared target rows [N+gamma-1, V] (pair (t,k) on row t+k): N={self.N} "
                    "positions x gamma=3, V=151936, bf16 logits, draft = target row + N(0,0.5), fp32 gradient, T=1")
        return (f"e2e TV loss fwd+bwd: N={self.N} positions x gamma=3, V=151936, bf16 logits (entropy-spanning target, "
                "draft = target + N(0,0.5)), fp32 gradient, T=1")


def method_stats(out) -> dict:
    """What the method computed in the last timed call, read back after the
    timed region: acceptance (mean accepted drafts per sequence, acceptance
    rate per draft position), the mean overlap alpha and target entropy, the
    TV loss, and how many rows came back flagged."""
    import numpy as np

    if out is None:
        return {}
    f = out._asdict()
    r = {}
    flags = f["row_flags"].cpu().numpy()
    good = flags == 0
    r["flagged_rows"] = int((~good).sum())
    if "accept_len" in f:
        n = f["accept_len"].cpu().numpy()[good]
        gamma = f["tokens"].shape[1] - 1
        r["mean_accept_len"] = float(n.mean()) if n.size else None
        r["acceptance_rate"] = float(n.mean() / gamma) if n.size else None
    if f.get("alpha") is not None:
        a = f["alpha"].cpu().numpy()[good]
        r["mean_alpha"] = float(np.nanmean(a)) if a.size else None
    ent = f.get("entropy", f.get("ent_p"))
    if ent is not None:
        e = ent.cpu().numpy()[good]
        r["mean_entropy_nats"] = float(np.nanmean(e)) if e.size else None
    if "rs_better" in f:
        rb = f["rs_better"].cpu().numpy()[good]
        r["rs_better_fraction"] = float(rb.mean()) if rb.size else None
    if "loss" in f:
        lo = f["loss"].cpu().numpy()[good]
        r["mean_loss"] = float(lo.mean()) if lo.size else None
    return r


def time_graph(wl, steps: int, warmup: int, device) -> dict:
    """Capture `copies` consecutive calls in a CUDA graph; replay; time K calls."""
    import torch

    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    for i in range(max(1, wl.copies)):
        wl.call(i)  # first calls: plan caches, output allocation
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        stream.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.graph(g, stream=stream):
            for i in range(wl.copies):
                wl.call(i, stream=torch.cuda.current_stream(device))
    torch.cuda.synchronize(device)
    reps, extra = divmod(steps, wl.copies)
    wreps = max(1, math.ceil(warmup / wl.copies))
    with torch.cuda.stream(stream):
        for _ in range(wreps):
            g.replay()
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        for i in range(extra):
            wl.call(i, stream=stream)
        ev1.record(stream)
    torch.cuda.synchronize(device)
    ms = ev0.elapsed_time(ev1)
    return {"ms_total": ms, "ms_per_step": ms / steps, "launches": steps}


def time_e2e(wl: VerifyWorkload, steps: int, warmup: int, device) -> dict:
    """Same metric through the public call with pinned host buffers: per step
    H2D of the inputs, the call, D2H of tokens and accept lengths.  Two input
    buffers: step i+1's inputs copy on a copy stream while step i runs (the
    way a caller keeps both the host link and the GPU busy)."""
    import torch

    host = [t.cpu().pin_memory() for t in wl.inputs[0]]
    dev_in = [[torch.empty_like(t) for t in wl.inputs[0]] for _ in range(2)]
    outs = [None, None]
    tok_h = torch.empty((2, wl.B, wl.gamma + 1), dtype=torch.int32).pin_memory()
    len_h = torch.empty((2, wl.B), dtype=torch.int32).pin_memory()
    copy_s, comp_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def h2d(i):
        j = i % 2
        copy_s.wait_event(freed[j])  # the call that last read buffer j is done
        with torch.cuda.stream(copy_s):
            for d, h in zip(dev_in[j], host):
                d.copy_(h, non_blocking=True)
        copied[j].record(copy_s)

    def run(i):
        j = i % 2
        comp_s.wait_event(copied[j])
        with torch.cuda.stream(comp_s):
            outs[j] = wl.mtp.mtp_rs_verify(*dev_in[j], with_stats=wl.stats, out=outs[j], stream=comp_s)
            freed[j].record(comp_s)
            tok_h[j].copy_(outs[j].tokens, non_blocking=True)
            len_h[j].copy_(outs[j].accept_len, non_blocking=True)

    for j in range(2):
        freed[j].record(comp_s)
    for i in range(warmup):
        h2d(i)
        run(i)
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(copy_s)
    comp_s.wait_event(ev0)
    h2d(0)
    for i in range(steps):
        if i + 1 < steps:
            h2d(i + 1)
        run(i)
    ev1.record(comp_s)
    torch.cuda.synchronize(device)
    ms = ev0.elapsed_time(ev1)
    h2d_b = sum(h.numel() * h.element_size() for h in host)
    d2h_b = tok_h[0].numel() * 4 + len_h[0].numel() * 4
    return {"value": wl.positions * steps / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d_b,
            "d2h_bytes_per_step": d2h_b, "steps": steps, "ms_per_step": ms / steps,
            "pipeline": "two input buffers; step i+1's host-to-device copy overlaps step i's call"}


# ------------------------------------------------------------ CPU oracle ---

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip() + f" ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def _oracle_pass(kind: str, x, n: int):
    """One oracle evaluation of the first n sequences (positions) of inputs x:
    verify (with statistics where the config asks), row statistics or the TV
    loss with its gradient."""
    import oracle

    if kind == "tv":
        oracle.tv_loss(x.target[:n], x.draft[:n], x.temperature, x.grad_scale)
    elif kind == "stats":
        oracle.row_stats(x.target[:n], x.draft[:n], x.temperature[:n])
    else:
        oracle.verify(x.target[:n], x.draft[:n], x.draft_ids[:n], x.temperature[:n], x.uniforms[:n],
                      want_stats=x.want_stats)


def oracle_rate(name: str, threads: int, n=None, min_s: float = 0.0, x=None, kind: str = None) -> dict:
    """Positions/s of the float64 oracle (as it stands) on `threads` host
    threads over the first n sequences (positions) of the named config, whole
    passes repeated until min_s seconds have passed (at least one pass)."""
    import oracle
    import workloads as W

    if x is None:
        x = W.config(name, N_override=512) if name == "tvloss" else W.config(name)
    kind = kind or ("tv" if name == "tvloss" else "verify")
    units = x.N if name == "tvloss" else x.B
    n = units if n is None else min(n, units)
    full = oracle.num_threads()
    oracle.set_threads(threads)
    try:
        _oracle_pass(kind, x, min(n, 2))  # page in the code and the first rows
        t0 = time.perf_counter()
        reps = 0
        while True:
            _oracle_pass(kind, x, n)
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                break
        used = oracle.num_threads()
    finally:
        oracle.set_threads(full)
    what = "positions" if name == "tvloss" else "sequences"
    if name == "tvloss":
        scope = f"subset: {n} positions drawn by the tvloss recipe on the host (the full config has 16384)"
    else:
        scope = "full config" if n == units else f"subset: the first {n} of {units} sequences"
    return {"value": reps * n * x.gamma / el, "unit": UNIT, "cores": used, "kind": "oracle", "seconds": el,
            "passes": reps, "sample": f"{scope}; {reps} pass(es) of {n} {what} in {el:.2f} s, float64 C, OpenMP"}


# timed workload -> (input config, oracle call, sequences or positions timed on
# all cores, on one core); None = the whole config
CPU_PLAN = {"tiny": ("tiny", "verify", None, None), "verify64": ("verify64", "verify", None, 8),
            "rl512": ("rl512", "verify", None, 32), "deep256": ("deep256", "verify", None, 8),
            "stats256": ("deep256", "stats", None, 8), "tvloss": ("tvloss", "tv", 512, 16)}


def cpu_baselines(headline: str, min_s: float, which: str) -> tuple:
    """The oracle timed on the host cores: the headline config in full,
    repeated for at least min_s seconds (the line's cpu_baseline), and with
    which == "all" every config of the plan on all cores and on one core."""
    import oracle
    import workloads as W

    allc = oracle.num_threads()
    model = cpu_model()
    head = oracle_rate(headline, allc, None, min_s)
    head["cpu_model"] = model
    table = None
    if which == "all":
        table = {"cpu_model": model, "cores_all": allc}
        inputs = {}
        for name, (cfg, kind, n_all, n_one) in CPU_PLAN.items():
            if cfg not in inputs:
                inputs[cfg] = W.config(cfg, N_override=n_all) if cfg == "tvloss" else W.config(cfg)
            x = inputs[cfg]
            table[name] = {"all_cores": oracle_rate(cfg, allc, n_all, 0.0, x=x, kind=kind),
                           "one_core": oracle_rate(cfg, 1, n_one, 0.0, x=x, kind=kind)}
        del inputs
    return head, table


# ------------------------------------------------------------------- main --

def run_reference(args, world, rank):
    """Reference arm: the float64 oracle timed on the host cores, on the
    headline workload (rl512), each step a bounded sample of its sequences."""
    if rank != 0:
        return
    import oracle
    import workloads as W

    x = W.config("rl512")
    sample = 32
    sl = slice(0, sample)
    a = (x.target[sl], x.draft[sl], x.draft_ids[sl], x.temperature[sl], x.uniforms[sl])
    for _ in range(args.warmup):
        oracle.verify(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify(*a)
    el = time.perf_counter() - t0
    val = args.steps * sample * x.gamma / el
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"rl512 (bounded sample: the first {sample} of 512 sequences per step)", "B": 512,
                   "gamma": 3, "V": 151936, "input_dtype": "bf16"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"the first {sample} sequences of rl512 per step", "cpu_model": cpu_model()},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_cuda(args, world, rank, local, pg):
    import torch

    import mtp_speculative_decoding_row_gb300 as mtp
    from mtp_speculative_decoding_row_gb300 import build as mtp_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or not os.path.exists(mtp_build.LIB):
        mtp_build.build()
    barrier(pg, device)
    mtp.load_library()
    if args.tv_kernel != "auto":
        mtp.mtp_set_tuning(tv_kernel={"tmem": mtp.KERNEL_TMEM, "stream": mtp.KERNEL_STREAM,
                                      "resident": mtp.KERNEL_RESIDENT}[args.tv_kernel])
    peaks = load_peaks()
    peak = peaks["hbm_gbs"]
    uuid = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"

    names = [w for w in args.workloads.split(",") if w]
    results = {}
    head = None
    for name in names:
        if name in TV_WORKLOADS:
            wl = TVWorkload(device, args.tv_n, shared=name == "tvshared", topk=name == "tvtopk")
            steps = max(3, min(args.steps, 20)) if name != names[0] else args.steps
        else:
            per_copy = VerifyWorkloadBytes(name)
            copies = max(2, math.ceil(4 * L2_BYTES / per_copy))
            wl = VerifyWorkload(name, device, min(copies, 8), args.deep_b)
            steps = args.steps
        sampler = ClockSampler(gpu_id) if name == names[0] else None
        barrier(pg, device)
        torch.cuda.synchronize(device)
        if sampler:
            sampler.start()
        torch.cuda.nvtx.range_push(f"mtp {name}")  # a range per workload for timeline tools
        t = time_graph(wl, steps, args.warmup, device)
        torch.cuda.nvtx.range_pop()
        clocks = sampler.stop() if sampler else None
        t_ms = max_over_ranks(pg, t["ms_total"], device)
        alg = wl.alg_bytes()
        per_launch_s = t["ms_total"] / 1e3 / t["launches"]
        achieved = alg / per_launch_s / 1e9
        tv = name in TV_WORKLOADS
        units = wl.N if tv else (wl.B * wl.gamma if wl.kind in ("sample", "gsample") else wl.B)  # draft sampling: rows
        if tv and name == "tvtopk":  # the top-K path runs on the streaming TV kernel
            with mtp.tuning(tv_kernel=mtp.KERNEL_STREAM):
                plan = mtp.mtp_query_plan("tv_loss", "bf16", units, wl.gamma, wl.V)
        else:
            plan = mtp.mtp_query_plan("tv_loss" if tv else wl.plan_op(), "bf16" if wl.es == 2 else "f32", units,
                                      wl.gamma, wl.V)
        r = {
            "workload": wl.describe(),
            "launch_plan": plan,
            "positions_per_s": world * wl.positions * steps / (t_ms / 1e3),
            "ms_per_step": t_ms / steps,
            "logit_gbps": achieved,
            "roofline_frac": achieved / peak,
            "alg_bytes_per_step": alg,
            "full_bytes_per_step": wl.bytes_full,
            "steps": steps,
            "input_copies": wl.copies,
        }
        r["traffic"] = traffic_for(name)
        r["method"] = method_stats(wl.out if tv else wl.outs[0])
        results[name] = r
        if head is None:
            head = (name, wl, t, t_ms, steps, clocks, alg, achieved)
        del wl
        torch.cuda.empty_cache()

    name, wl0, t, t_ms, steps, clocks, alg, achieved = head
    # e2e leg on the headline workload
    e2e = None
    if name not in TV_WORKLOADS:
        wl = VerifyWorkload(name, device, 1)
        e2e = time_e2e(wl, max(3, min(args.steps, 50)), max(3, args.warmup), device)
        e2e["value"] = max_over_ranks(pg, -e2e["value"], device) * -1 * world
    h = csrc_hash()
    traffic_val = traffic_for(name)
    cpu, cpu_table = None, None
    if rank == 0 and world == 1 and args.cpu_baselines != "none" and name not in TV_WORKLOADS:
        cpu, cpu_table = cpu_baselines(name, args.cpu_seconds, args.cpu_baselines)

    if cpu_table:
        for wname, r in results.items():
            if wname in CPU_PLAN:
                r["cpu_baseline"] = cpu_table[wname]
    if rank == 0:
        hr = results[name]
        line = {
            "metric": METRIC, "value": hr["positions_per_s"], "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": hr["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "input_dtype": "bf16" if wl0.es == 2 else "f32",
            "dtype_note": "dtype is the arithmetic type; input_dtype is the logits' storage", "data": "synthetic",
            "config": {"workload": hr["workload"], "B": wl0.B if hasattr(wl0, "B") else wl0.N, "gamma": wl0.gamma,
                       "V": wl0.V, "input_dtype": "bf16" if wl0.es == 2 else "f32",
                       "l2": f"{hr['input_copies']} rotated input copies of {hr['full_bytes_per_step'] / 1e6:.0f} MB "
                             f"(> 4x L2 between reuses)",
                       "timing": "CUDA graph replay, CUDA events on the launching stream",
                       "parallelism": f"replicas x{world}"},
            "logit_gbps": hr["logit_gbps"],
            "logit_gbps_full_rows": hr["full_bytes_per_step"] / (hr["ms_per_step"] / 1e3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic_val,
                         "peak_source": f"{peaks['source']} hbm_gbs (MEASURED_PEAKS.json)",
                         "algorithmic_bytes_per_launch": alg},
            "cpu_baseline": cpu,
            "cpu_baselines": cpu_table,
            "e2e": e2e,
            "gpu_launches": t["launches"],
            "clocks": clocks,
            "workloads": results,
            "kernel_sources": h,
        }
        print(json.dumps(line), flush=True)


def VerifyWorkloadBytes(name: str) -> int:
    return {"verify64": 64 * 7 * 151936 * 2, "rl512": 512 * 7 * 151936 * 2, "deep256": 256 * 15 * 151936 * 4,
            "stats256": 256 * 15 * 151936 * 4, "diag256": 256 * 15 * 151936 * 4, "to64": 64 * 7 * 151936 * 2,
            "gumbel64": 64 * 7 * 151936 * 2, "sample192": 192 * 151936 * 2, "gsample192": 192 * 151936 * 2}[name]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workloads", default="rl512,verify64,deep256,stats256,diag256,to64,gumbel64,sample192,"
                                           "gsample192,tvloss,tvshared,tvtopk")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum seconds of oracle time for the headline cpu_baseline")
    ap.add_argument("--cpu-baselines", choices=["all", "headline", "none"], default="all",
                    help="oracle timings: every config on all cores and one core, the headline only, or none")
    ap.add_argument("--tv-n", type=int, default=None, help="TV-loss positions (default 16384; smaller for profiling)")
    ap.add_argument("--tv-kernel", choices=["auto", "tmem", "stream", "resident"], default="auto",
                    help="TV-loss kernel (the library's tuning API; auto = the planner's choice)")
    ap.add_argument("--deep-b", type=int, default=None,
                    help="sequences of the deep256-based workloads (default 256; smaller for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_cuda(args, world, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
