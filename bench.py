#!/usr/bin/env python3
"""Benchmark of the shifted-window block-glue hot path on GB300.

One step = one pass of every kernel of the path over the Pangu-Weather
stage shapes, ten launches:
  ln_fwd, residual_add_ln_fwd, window_gather, norm_gather at
      C=192: 131040 tokens (8x91x180), 138240 windowed rows (8x96x180)
      C=384:  32760 tokens (4x91x90),   34560 windowed rows (4x96x90)
  bias_gelu_tanh fp32 [131040, 768] and fp16 [32760, 1536]
Window (2,6,12), shift (1,3,6).  Inputs are seeded synthetic tensors.

Metric: effective HBM GB/s (algorithmic bytes: each input read once, each
output written once, plus the index array) and ms per call per kernel.
Beyond the step the line carries the other rows of the path (block-boundary
fusions, the C=384 gathers over whole windows, bfloat16 forms, the GELU
backward, the attention bias-mask add), a GELU rows sweep (1k-256k rows),
the end-to-end figure from pinned host memory, the oracle's rate on the
host CPU (one thread on a quarter of the rows, and all cores on every row),
and, as its last two keys, the LayerNorm-family kernels' figures
(headline_kernels) and the parity gate: every output element the timed
buffers hold, read back after timing and compared with the oracle's.
A step's ten launches are captured once, through the public API, in a CUDA
graph; the graph is replayed K times back to back and CUDA events on the
launching stream bracket the K replays.  One step touches 1.77 GB (13x the
L2), so every input is read from HBM and earlier outputs drain to HBM while
later kernels run.  Per-kernel ms/call comes from each kernel alone,
replayed back to back over rotating buffer sets.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (independent
replicas, no collective on the data path); the line reports the sum of the
ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from window_gather_swin_gb300 import synth  # noqa: E402

METRIC = "effective HBM GB/s and ms/call per fused kernel at [131040,192]/[32760,384]"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
EPS = 1e-5
CPU_SAMPLE_FRACTION = 0.25


# ------------------------------------------------------------ workload ----

class Call:
    """One kernel invocation of the step with its inputs, outputs and bytes."""

    def __init__(self, name, workload, nbytes, inputs, outputs, run, oracle, rows):
        self.name = name
        self.workload = workload
        self.bytes = int(nbytes)
        self.inputs = inputs        # {key: cpu tensor}
        self.outputs = outputs      # {key: (shape, dtype)}
        self.run = run              # run(dev_inputs, dev_outputs)
        self.oracle = oracle        # OracleLeg of the call, or None
        self.rows = rows

    @property
    def label(self):
        return f"{self.name} {self.workload}"


class OracleLeg:
    """The oracle's side of one call, over a range [lo, hi) of its `units`
    (token rows, or destination rows for the gathers):
      compute(lo, hi) -> the oracle's outputs for those units (what is timed);
      nbytes(lo, hi)  -> their algorithmic bytes;
      check(gpu, orc, lo, hi) -> statistics of the GPU outputs of the same
          units against the oracle's under the parity rules of
          tests/parity.py; raises AssertionError on a violation.
    The oracle legs build their window maps with the oracle's own builder,
    so nothing here calls into the CUDA library."""

    def __init__(self, units, compute, nbytes, check):
        self.units = units
        self.compute = compute
        self.nbytes = nbytes
        self.check = check


# The workload both arms report: the ten launches of one step.
STEP_CONFIG = {
    "workload": ("block-glue hot path, both stages: ln, residual_add_ln, window_gather, "
                 "norm_gather at [131040,192]->138240 and [32760,384]->34560; bias_gelu fp32 "
                 "[131040,768], fp16 [32760,1536]"),
    "window": list(synth.WINDOW), "shift": list(synth.SHIFT),
}


def _orc():
    # The oracle is test infrastructure; only the CPU legs of this benchmark
    # (cpu_baseline, the parity gate and the reference arm) execute it.
    import oracle
    return oracle


def _rules():
    # the comparison rules of the GPU parity tests, for the parity gate
    from tests import parity
    return parity


def _oracle_map(st):
    return _orc().build_window_index(st.grid, synth.WINDOW, synth.SHIFT, st.padded)


def _ln_leg(x, n, c):
    x = x.numpy()

    def check(g, o, lo, hi):
        return {"ln": _rules().check_ln(g["y"], o["y"], _orc().ln_f64(x[lo:hi], EPS), "ln_fwd")}
    return OracleLeg(n, lambda lo, hi: {"y": _orc().ln(x[lo:hi], EPS)},
                     lambda lo, hi: 4 * (hi - lo) * c, check)


def _add_ln_leg(a, b, n, c):
    a, b = a.numpy(), b.numpy()

    def compute(lo, hi):
        r, y = _orc().residual_add_ln(a[lo:hi], b[lo:hi], EPS)
        return {"r": r, "y": y}

    def check(g, o, lo, hi):
        _rules().assert_bitwise(g["r"], o["r"], "residual_out")
        return {"bitwise": g["r"].size,
                "ln": _rules().check_ln(g["y"], o["y"], _orc().ln_f64(o["r"], EPS), "add_ln y")}
    return OracleLeg(n, compute, lambda lo, hi: 8 * (hi - lo) * c, check)


def _gather_leg(src, st, norm):
    src = src.numpy()
    n, c = src.shape
    idx = _oracle_map(st)
    m = idx.size

    def compute(lo, hi):
        if norm:
            dst, bad = _orc().norm_gather(src, idx[lo:hi], EPS)
        else:
            dst, bad = _orc().window_gather(src, idx[lo:hi])
        return {"dst": dst, "bad": bad}

    def check(g, o, lo, hi):
        assert o["bad"] == 0, "the oracle's own map holds an index outside [-1, n_src)"
        if not norm:
            _rules().assert_bitwise(g["dst"], o["dst"], "window_gather")
            return {"bitwise": g["dst"].size}
        i = idx[lo:hi]
        pad = i < 0
        _rules().assert_bitwise(g["dst"][pad], o["dst"][pad], "norm_gather pad rows")
        assert not o["dst"][pad].view(np.uint16).any(), "oracle pad rows are not zero"
        ln = _rules().check_ln(g["dst"][~pad], o["dst"][~pad], _orc().ln_f64(src[i[~pad]], EPS),
                               "norm_gather")
        return {"bitwise": g["dst"][pad].size, "ln": ln}
    return OracleLeg(m, compute, lambda lo, hi: (hi - lo) / m * (2 * c * n) + (hi - lo) * (2 * c + 4),
                     check)


def _gelu_leg(x, b, rows, width, esz):
    x, b = x.numpy(), b.numpy()

    def compute(lo, hi):
        return {"y": _orc().bias_gelu_tanh(x[lo:hi], b, want_f64=False)[0]}

    def check(g, o, lo, hi):
        y, y64 = _orc().bias_gelu_tanh(x[lo:hi], b, want_f64=True)  # unrounded values
        assert np.array_equal(y.view(np.uint8), o["y"].view(np.uint8)), "oracle not repeatable"
        if esz == 4:
            return {"gelu_f32": _rules().check_gelu_f32(g["y"], y64, "bias_gelu fp32")}
        return {"gelu_f16": _rules().check_fp16_near(g["y"], y, y64, "bias_gelu fp16")}
    return OracleLeg(rows, compute, lambda lo, hi: 2 * (hi - lo) * width * esz + width * esz, check)


def build_calls(gpu=True):
    """The ten calls of one step.  With gpu=False (the reference arm) the
    index maps come from the oracle's builder and nothing touches the CUDA
    library; the maps are identical either way."""
    import window_gather_swin_gb300 as wgs
    calls = []
    for st in (synth.STAGE_192, synth.STAGE_384):
        n, c = st.tokens, st.width
        x = synth.ln_input(n, c, seed=1)
        calls.append(Call(
            "ln_fwd", f"[{n},{c}]", 4 * n * c, {"x": x}, {"y": ((n, c), torch.float16)},
            lambda i, o: wgs.ln_fwd(i["x"], EPS, out=o["y"]), _ln_leg(x, n, c), n))
        a, b = synth.residual_branch(n, c, seed=2)
        calls.append(Call(
            "residual_add_ln_fwd", f"[{n},{c}]", 8 * n * c, {"a": a, "b": b},
            {"r": ((n, c), torch.float16), "y": ((n, c), torch.float16)},
            lambda i, o: wgs.residual_add_ln_fwd(i["a"], i["b"], EPS, residual_out=o["r"], out=o["y"]),
            _add_ln_leg(a, b, n, c), n))
        src = synth.gather_source(n, c, seed=3)
        if gpu:
            idx = wgs.build_window_index(st.grid, synth.WINDOW, synth.SHIFT, st.padded)
        else:
            idx = torch.from_numpy(_oracle_map(st))
        m = idx.numel()
        gbytes = 2 * c * n + 2 * c * m + 4 * m
        for name in ("window_gather", "norm_gather"):
            if name == "window_gather":
                run = lambda i, o: wgs.window_gather(i["src"], i["idx"], out=o["dst"])
            else:
                run = lambda i, o: wgs.norm_gather(i["src"], i["idx"], EPS, out=o["dst"])
            calls.append(Call(
                name, f"[{n},{c}]->{m}", gbytes, {"src": src, "idx": idx},
                {"dst": ((m, c), torch.float16)}, run,
                _gather_leg(src, st, norm=name == "norm_gather"), m))
    for (rows, width), dt, seed in ((synth.GELU_F32_SHAPE, torch.float32, 4),
                                    (synth.GELU_F16_SHAPE, torch.float16, 4)):
        x, b = synth.gelu_input(rows, width, dt, seed=seed)
        esz = 4 if dt == torch.float32 else 2
        calls.append(Call(
            "bias_gelu_tanh", f"{'fp32' if esz == 4 else 'fp16'} [{rows},{width}]",
            2 * rows * width * esz + width * esz, {"x": x, "bias": b},
            {"y": ((rows, width), dt)},
            lambda i, o: wgs.bias_gelu_tanh(i["x"], i["bias"], out=o["y"]),
            _gelu_leg(x, b, rows, width, esz), rows))
    return calls


def build_next_calls():
    """The rows beyond the step: the block-boundary fusions (window reverse +
    residual add + LN; residual add + norm1 + window gather) at both stages,
    the bfloat16 forms, the GELU backward and the attention bias-mask add."""
    import window_gather_swin_gb300 as wgs
    calls = []
    for st in (synth.STAGE_192, synth.STAGE_384):
        n, c = st.tokens, st.width
        idx = wgs.build_window_index(st.grid, synth.WINDOW, synth.SHIFT, st.padded)
        inv = wgs.build_window_inverse(st.grid, synth.WINDOW, synth.SHIFT, st.padded)
        m = idx.numel()
        res, br = synth.residual_branch(n, c, seed=2)
        windows = synth.gather_source(m, c, seed=3)
        calls.append(Call(
            "window_reverse_add_ln_fwd", f"{m}->[{n},{c}]", 8 * n * c + 4 * n,
            {"res": res, "win": windows, "inv": inv},
            {"r": ((n, c), torch.float16), "y": ((n, c), torch.float16)},
            lambda i, o: wgs.window_reverse_add_ln_fwd(i["res"], i["win"], i["inv"], EPS,
                                                       residual_out=o["r"], out=o["y"]),
            None, n))
        calls.append(Call(
            "residual_add_norm_gather", f"[{n},{c}]->{m}", 6 * n * c + (2 * c + 4) * m,
            {"a": res, "b": br, "idx": idx},
            {"r": ((n, c), torch.float16), "dst": ((m, c), torch.float16)},
            lambda i, o: wgs.residual_add_norm_gather(i["a"], i["b"], i["idx"], EPS,
                                                      residual_out=o["r"], out=o["dst"]),
            None, m))
    # C = 384 with whole windows (4x96x96, 36864 rows): the map a block at
    # that stage uses end to end, since its attention needs equal windows
    st = synth.STAGE_384
    n, c = st.tokens, st.width
    idx = wgs.build_window_index(st.grid, synth.WINDOW, synth.SHIFT, synth.ATTN_384.padded)
    m = idx.numel()
    src = synth.gather_source(n, c, seed=3)
    calls.append(Call("window_gather", f"[{n},{c}]->{m}", 2 * c * n + (2 * c + 4) * m,
                      {"src": src, "idx": idx}, {"dst": ((m, c), torch.float16)},
                      lambda i, o: wgs.window_gather(i["src"], i["idx"], out=o["dst"]), None, m))
    calls.append(Call("norm_gather", f"[{n},{c}]->{m}", 2 * c * n + (2 * c + 4) * m,
                      {"src": src, "idx": idx}, {"dst": ((m, c), torch.float16)},
                      lambda i, o: wgs.norm_gather(i["src"], i["idx"], EPS, out=o["dst"]), None, m))
    # bfloat16 forms at the large stage / MLP width
    st = synth.STAGE_192
    n, c = st.tokens, st.width
    bf = torch.bfloat16
    xb = synth.ln_input(n, c, seed=1, dtype=bf)
    calls.append(Call("ln_fwd", f"bf16 [{n},{c}]", 4 * n * c, {"x": xb},
                      {"y": ((n, c), bf)}, lambda i, o: wgs.ln_fwd(i["x"], EPS, out=o["y"]),
                      None, n))
    idx = wgs.build_window_index(st.grid, synth.WINDOW, synth.SHIFT, st.padded)
    m = idx.numel()
    ab, bb = synth.residual_branch(n, c, seed=2, dtype=bf)
    calls.append(Call(
        "residual_add_norm_gather", f"bf16 [{n},{c}]->{m}", 6 * n * c + (2 * c + 4) * m,
        {"a": ab, "b": bb, "idx": idx}, {"r": ((n, c), bf), "dst": ((m, c), bf)},
        lambda i, o: wgs.residual_add_norm_gather(i["a"], i["b"], i["idx"], EPS,
                                                  residual_out=o["r"], out=o["dst"]),
        None, m))
    calls.append(Call(
        "residual_add_ln_fwd", f"bf16 [{n},{c}]", 8 * n * c, {"a": ab, "b": bb},
        {"r": ((n, c), bf), "y": ((n, c), bf)},
        lambda i, o: wgs.residual_add_ln_fwd(i["a"], i["b"], EPS, residual_out=o["r"], out=o["y"]),
        None, n))
    srcb = synth.gather_source(n, c, seed=3, dtype=bf)
    calls.append(Call(
        "norm_gather", f"bf16 [{n},{c}]->{m}", 2 * c * n + (2 * c + 4) * m,
        {"src": srcb, "idx": idx}, {"dst": ((m, c), bf)},
        lambda i, o: wgs.norm_gather(i["src"], i["idx"], EPS, out=o["dst"]), None, m))
    invb = wgs.build_window_inverse(st.grid, synth.WINDOW, synth.SHIFT, st.padded)
    winb = synth.gather_source(m, c, seed=3, dtype=bf)
    calls.append(Call(
        "window_reverse_add_ln_fwd", f"bf16 {m}->[{n},{c}]", 8 * n * c + 4 * n,
        {"res": ab, "win": winb, "inv": invb}, {"r": ((n, c), bf), "y": ((n, c), bf)},
        lambda i, o: wgs.window_reverse_add_ln_fwd(i["res"], i["win"], i["inv"], EPS,
                                                   residual_out=o["r"], out=o["y"]),
        None, n))
    rows, width = synth.GELU_F16_SHAPE
    xg, bg = synth.gelu_input(rows, width, bf, seed=4)
    # backward of bias + GELU (algorithmic bytes: grad_y and x read, grad_x
    # written, bias read and grad_bias written; the partial sums are extra)
    for (r_, w_), dt_ in ((synth.GELU_F32_SHAPE, torch.float32), (synth.GELU_F16_SHAPE, torch.float16),
                          (synth.GELU_F16_SHAPE, bf)):
        esz = 4 if dt_ == torch.float32 else 2
        tag = {torch.float32: "fp32", torch.float16: "fp16", bf: "bf16"}[dt_]
        xg_, bg_ = synth.gelu_input(r_, w_, dt_, seed=4)
        gy_, _ = synth.gelu_input(r_, w_, dt_, seed=5)
        calls.append(Call(
            "bias_gelu_tanh_bwd", f"{tag} [{r_},{w_}]",
            3 * r_ * w_ * esz + 2 * w_ * esz, {"gy": gy_, "x": xg_, "bias": bg_},
            {"gx": ((r_, w_), dt_), "gb": ((w_,), dt_), "ws": ((wgs.gelu_bwd_workspace_bytes(r_, w_),), torch.uint8)},
            lambda i, o: wgs.bias_gelu_tanh_bwd(i["gy"], i["x"], i["bias"], grad_x=o["gx"],
                                                grad_bias=o["gb"], workspace=o["ws"]),
            None, r_))
    calls.append(Call("bias_gelu_tanh", f"bf16 [{rows},{width}]", 4 * rows * width + 2 * width,
                      {"x": xg, "bias": bg}, {"y": ((rows, width), bf)},
                      lambda i, o: wgs.bias_gelu_tanh(i["x"], i["bias"], out=o["y"]), None, rows))
    # position bias + shift mask on the attention logits (algorithmic bytes:
    # logits read and written, the bias slab and the labels read once)
    for ast, dt_ in ((synth.ATTN_192, torch.float16), (synth.ATTN_384, torch.float16),
                     (synth.ATTN_192, bf)):
        s_, b_ = synth.attention_logits(ast.n_win, ast.heads, ast.n, 1, seed=6, dtype=dt_)
        reg = wgs.build_shift_regions(ast.grid, synth.WINDOW, synth.SHIFT, ast.padded)
        tag = "fp16" if dt_ == torch.float16 else "bf16"
        calls.append(Call(
            "window_bias_mask_add", f"{tag} [{ast.n_win},{ast.heads},{ast.n},{ast.n}]",
            4 * s_.numel() + 2 * b_.numel() + 4 * reg.numel(),
            {"s": s_, "b": b_, "reg": reg}, {"out": (tuple(s_.shape), dt_)},
            lambda i, o: wgs.window_bias_mask_add(i["s"], i["b"], None, i["reg"], out=o["out"]),
            None, ast.n_win * ast.heads * ast.n))
    return calls


# ---------------------------------------------------------------- util ----

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic():
    """dram bytes per launch from ncu captures, keyed by kernel label.  Each
    line of profiles/ncu_traffic.txt is `label | sources digest | bytes`; a
    figure counts only while the sources of that kernel still hash to its
    digest (see sources_digest)."""
    out = {}
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return out
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line.count("|") != 2:
                continue
            label, sha, nbytes = (p.strip() for p in line.split("|"))
            if sha == sources_digest(label):
                out[label] = float(nbytes)
    return out


KERNEL_SOURCES = {  # first matching prefix wins
    "bias_gelu_tanh_bwd": ["window_gather_swin_gb300/csrc/wgs_gelu_bwd.cu"],
    "bias_gelu_tanh": ["window_gather_swin_gb300/csrc/wgs_gelu.cu"],
    "window_bias_mask_add": ["window_gather_swin_gb300/csrc/wgs_bias_mask.cu"],
    "": ["window_gather_swin_gb300/csrc/wgs_rows.cu"],  # LN, add + LN, gathers
}


def sources_digest(label: str) -> str:
    """Hash of the files that define the kernel behind `label`: its .cu file
    and the shared device header (the C ABI header only declares)."""
    import hashlib
    own = next(v for k, v in KERNEL_SOURCES.items() if label.startswith(k))
    files = own + ["window_gather_swin_gb300/csrc/wgs_common.cuh"]
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        deadline = time.time() + 3.0
        while not self.lines and time.time() < deadline:  # first sample is in
            time.sleep(0.01)
        self.mark = len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(self.interval_ms / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l.split(",") for _, l in self.lines[max(self.mark - 1, 0):]]
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        sm = [float(r[1]) for r in rows if _num(r[1])]
        mx = [float(r[2]) for r in rows if _num(r[2])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _num(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# ------------------------------------------------------------ our arm ----

def host_cpu():
    """Cores this process may run on, and the host CPU's model name."""
    cores = len(os.sched_getaffinity(0))
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return cores, model


def _ranges(n, parts):
    step = max(1, -(-n // parts))
    return [(lo, min(n, lo + step)) for lo in range(0, n, step)]


def oracle_step(calls, threads, fraction=1.0):
    """The oracle, as it stands, on the first `fraction` of the units of
    every call of `calls`.  With threads > 1 each call's units are split
    into row ranges run on that many host threads (the oracle's C code runs
    outside the GIL).  Returns (seconds, algorithmic bytes, outputs), where
    outputs[j] lists ((lo, hi), oracle outputs) of call j; only the oracle
    calls are timed."""
    secs = nbytes = 0.0
    outs = []
    ex = ThreadPoolExecutor(threads) if threads > 1 else None
    try:
        for c in calls:
            leg = c.oracle
            k = max(1, int(leg.units * fraction))
            parts = _ranges(k, threads * 4) if ex else [(0, k)]
            t0 = time.perf_counter()
            res = list(ex.map(lambda r: leg.compute(*r), parts)) if ex else [leg.compute(0, k)]
            secs += time.perf_counter() - t0
            nbytes += leg.nbytes(0, k)
            outs.append(list(zip(parts, res)))
    finally:
        if ex:
            ex.shutdown()
    return secs, nbytes, outs


def cpu_legs(calls, gpu_outs, want_baseline, want_parity):
    """The oracle on this host's CPU: Run 1 (one thread, the first quarter
    of every call's units: the cpu_baseline value), Run 2 (every unit, split
    over all usable cores, three repetitions, median) and the parity gate
    (every output element the timed buffers hold against Run 2's outputs)."""
    cores, model = host_cpu()
    keep = [j for j, c in enumerate(calls) if c.oracle is not None]
    calls = [calls[j] for j in keep]
    if gpu_outs is not None:
        gpu_outs = [gpu_outs[j] for j in keep]
    if not calls:
        return None, None
    base = parity = None
    last = None
    if want_baseline:
        s1, b1, _ = oracle_step(calls, 1, CPU_SAMPLE_FRACTION)
        reps = []
        for _ in range(3):
            s2, b2, last = oracle_step(calls, cores, 1.0)
            reps.append(s2)
        med = statistics.median(reps)
        base = {"value": round(b1 / s1 / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": (f"first {CPU_SAMPLE_FRACTION:g} of the units of each of the {len(calls)} "
                           f"calls of one step ({b1 / 1e6:.1f} MB algorithmic, {s1:.2f} s), one thread"),
                "sample_fraction": CPU_SAMPLE_FRACTION,
                "host_cores": cores, "cpu_model": model,
                "run2_all_cores": {"value": round(b2 / med / 1e9, 4), "unit": "GB/s",
                                   "cores": cores, "repetitions": len(reps),
                                   "s_median": round(med, 3), "s_min": round(min(reps), 3),
                                   "sample": "every unit of every call of one step"}}
    if want_parity and gpu_outs is not None:
        if last is None:
            _, _, last = oracle_step(calls, cores, 1.0)
        parity = parity_gate(calls, gpu_outs, last, cores)
    return base, parity


def parity_gate(calls, gpu_outs, orc_outs, threads):
    """Element-by-element comparison of the GPU outputs of `calls` with the
    oracle's, range by range, under the rules of tests/parity.py: identical
    bits for residual_out, gathered and pad rows; LayerNorm outputs inside
    the FP32 error bound and the 2e-3 bar (bar exceptions only as one-spacing
    flips at a rounding midpoint); fp32 GELU within 1e-5 relative; fp16 GELU
    inside the FP32 error bound."""
    tot = {"bitwise": 0, "ln_n": 0, "ln_max_abs": 0.0, "ln_tie_flips": 0, "ln_err_over_bound": 0.0,
           "gelu_f32_n": 0, "gelu_f32_max_rel": 0.0, "gelu_f16_n": 0, "gelu_f16_max_ulp": 0,
           "gelu_f16_err_over_bound": 0.0}
    failures = []

    def one(j, lo, hi, o):
        g = {k: v[lo:hi] for k, v in gpu_outs[j].items()}
        return calls[j].oracle.check(g, o, lo, hi)

    jobs = [(j, lo, hi, o) for j in range(len(calls)) for (lo, hi), o in orc_outs[j]]
    with ThreadPoolExecutor(threads) as ex:
        futs = [(calls[j].label, ex.submit(one, j, lo, hi, o)) for j, lo, hi, o in jobs]
        for label, f in futs:
            try:
                st = f.result()
            except AssertionError as e:
                failures.append(f"{label}: {str(e)[:300]}")
                continue
            tot["bitwise"] += int(st.get("bitwise", 0))
            if "ln" in st:
                ln = st["ln"]
                tot["ln_n"] += ln["n"]
                tot["ln_max_abs"] = max(tot["ln_max_abs"], ln["max_abs"])
                tot["ln_tie_flips"] += ln.get("above_abs_tol_tie_flips", 0)
                tot["ln_err_over_bound"] = max(tot["ln_err_over_bound"], ln["max_err_over_bound"])
            if "gelu_f32" in st:
                tot["gelu_f32_n"] += st["gelu_f32"]["n"]
                tot["gelu_f32_max_rel"] = max(tot["gelu_f32_max_rel"], st["gelu_f32"]["max_rel"])
            if "gelu_f16" in st:
                gf = st["gelu_f16"]
                tot["gelu_f16_n"] += gf["n"]
                tot["gelu_f16_max_ulp"] = max(tot["gelu_f16_max_ulp"], gf["max_ulp"])
                tot["gelu_f16_err_over_bound"] = max(tot["gelu_f16_err_over_bound"],
                                                     gf["max_err_over_bound"])
    elements = tot["bitwise"] + tot["ln_n"] + tot["gelu_f32_n"] + tot["gelu_f16_n"]
    out = {"pass": not failures, "elements": elements, "bitwise": tot["bitwise"],
           "ln": {"n": tot["ln_n"], "max_abs": tot["ln_max_abs"], "tie_flips": tot["ln_tie_flips"],
                  "err_over_bound": round(tot["ln_err_over_bound"], 4)},
           "gelu_f32": {"n": tot["gelu_f32_n"], "max_rel": tot["gelu_f32_max_rel"]},
           "gelu_f16": {"n": tot["gelu_f16_n"], "max_ulp": tot["gelu_f16_max_ulp"],
                        "err_over_bound": round(tot["gelu_f16_err_over_bound"], 4)},
           "scope": (f"every output element of the {len(calls)} timed calls, read back from the "
                     "timed buffers, against the oracle (rules of tests/parity.py)")}
    if failures:
        out["failures"] = failures[:5]
    return out


HEADLINE = ("ln_fwd", "residual_add_ln_fwd", "window_gather", "norm_gather")


def headline_kernels(kernels):
    """The LayerNorm-family step kernels at both stages, compactly: per
    kernel [us per call, GB/s, fraction of the measured copy peak, fraction
    of the nominal 8 TB/s]."""
    out = {"fields": ["us_per_call", "GB/s", "of_measured_peak", "of_8TB/s"]}
    for k in kernels:
        if k["kernel"] in HEADLINE and not k["workload"].startswith("bf16"):
            out[f"{k['kernel']} {k['workload']}"] = [round(k["ms_per_call"] * 1e3, 2), k["gbs"],
                                                     k["frac_of_measured"], k["frac_of_nominal_8tbs"]]
    return out


def capture(fn, dev):
    """Record the launches fn() makes into a CUDA graph (captured on a side
    stream after one eager warm-up there), so that replays run them back to
    back with no host work between launches."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize(dev)
    return g


def device_sets(calls, dev, n_sets):
    return [([{k: v.to(dev) for k, v in c.inputs.items()} for c in calls],
             [{k: torch.empty(sh, dtype=d, device=dev) for k, (sh, d) in c.outputs.items()}
              for c in calls]) for _ in range(n_sets)]


def run_ours(args, rank, world, local):
    import window_gather_swin_gb300 as wgs  # noqa: F401  (loads libwgs.so)
    from window_gather_swin_gb300 import _capi
    _capi.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    calls = build_calls()
    if args.only:
        want = args.only
        calls = [c for c in calls + build_next_calls()
                 if (c.label == want[1:] if want.startswith("=") else want in c.label)]
        if not calls:
            raise SystemExit(f"--only {args.only!r} matches no call")
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 128 * 2 ** 20)
    step_bytes = sum(c.bytes for c in calls)
    peak, peak_src = measured_hbm_peak()
    # Every input must come from HBM: consecutive uses of one buffer are
    # separated by at least 3x L2 of other traffic.  The full step touches
    # 1.77 GB, so one buffer set suffices; a subset (--only) rotates copies.
    n_sets = max(1, -(-3 * l2 // step_bytes))
    sets = device_sets(calls, dev, n_sets)
    stream = torch.cuda.current_stream(dev)

    def step(s, marks=None):
        dev_in, dev_out = sets[s % n_sets]
        if marks is not None:
            marks[0].record(stream)
        for j, (c, i, o) in enumerate(zip(calls, dev_in, dev_out)):
            c.run(i, o)
            if marks is not None:
                marks[j + 1].record(stream)

    # One graph per buffer set holds one step: the ten launches, back to back.
    graphs = [capture(lambda s=s: step(s), dev) for s in range(n_sets)]
    for s in range(args.warmup):  # untimed
        graphs[s % n_sets].replay()
    torch.cuda.synchronize(dev)

    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(smi_id(dev))
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    t0.record(stream)
    for s in range(K):
        graphs[s % n_sets].replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    barrier(world)
    clocks = sampler.stop()
    # the outputs the timed replays left in buffer set 0, for the parity gate
    gpu_outs = None
    if rank == 0 and not args.no_parity:
        gpu_outs = [{k: v.cpu().numpy() for k, v in o.items()} if c.oracle else None
                    for c, o in zip(calls, sets[0][1])]
    region_ms = t0.elapsed_time(t1)
    max_region_ms = reduce_max(region_ms, world, dev)
    all_bytes = reduce_sum(step_bytes * K, world, dev)
    value = all_bytes / (max_region_ms / 1e3) / 1e9
    del graphs

    # Per kernel, alone: the ms/call figures and the roofline.
    kernels = run_isolated(calls, dev, l2, peak, args.isolated_launches)
    dom = max(range(len(calls)), key=lambda j: kernels[j]["ms_per_call"])
    traffic = ncu_traffic().get(calls[dom].label)
    roofline = {"bound": "hbm", "kernel": calls[dom].label,
                "achieved": kernels[dom]["gbs"], "peak": peak, "unit": "GB/s",
                "frac": round(kernels[dom]["gbs"] / peak, 4), "peak_source": peak_src,
                "traffic": traffic, "algorithmic_bytes": calls[dom].bytes}

    kernels_next = sweep = None
    if not args.only:
        kernels_next = run_isolated(build_next_calls(), dev, l2, peak, args.isolated_launches)
        if not args.no_sweep:
            sweep = gelu_rows_sweep(dev, l2, peak, args.isolated_launches)

    # Diagnostic: the same step launched eagerly with an event between
    # launches, which attributes the step's time to its kernels (each also
    # drains its predecessor's dirty L2 lines here).
    in_step = None
    if not args.no_attribution:
        ka = min(K, 200)
        for s in range(3):
            step(s)
        marks = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
                 for _ in range(ka)]
        torch.cuda.synchronize(dev)
        for s in range(ka):
            step(s, marks[s])
        torch.cuda.synchronize(dev)
        in_step = []
        for j, c in enumerate(calls):
            p = [marks[s][j].elapsed_time(marks[s][j + 1]) for s in range(ka)]
            in_step.append({"kernel": c.name, "workload": c.workload,
                            "ms_mean": round(statistics.fmean(p), 5),
                            "ms_median": round(statistics.median(p), 5)})
    del sets

    e2e = None if args.no_e2e else run_e2e(calls, dev, args, world)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup,
        "ms_per_step": round(max_region_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "storage_dtype": "fp16 rows (LN, gathers, fp16 GELU), fp32 (fp32 GELU)",
        "data": "synthetic (seeded N(0,1)-family tensors of the stage shapes)",
        "config": step_config(world, args.only, len(calls), step_bytes=step_bytes, n_sets=n_sets),
        "l2": (f"inputs larger than L2: steps run back to back and one step touches "
               f"{step_bytes * n_sets / 1e6:.0f} MB over {n_sets} buffer set(s) "
               f"(L2 {l2 / 1e6:.0f} MB), so every input is read from HBM; no flush"),
        "timing": ("each step's launches are captured once in a CUDA graph through the "
                   "public API and replayed K times; CUDA events around the K replays on "
                   "the launching stream; value = all ranks' algorithmic bytes / slowest "
                   "rank's region time"),
        "wall_s": round(wall, 3),
        "kernels": kernels,
        "kernels_in_step": in_step,
        "kernels_next": kernels_next,
        "gelu_rows_sweep": sweep,
        "roofline": roofline,
        "gpu": {"name": torch.cuda.get_device_name(dev), "sms": props.multi_processor_count,
                "l2_bytes": l2, "cc": f"{props.major}.{props.minor}"},
        "clocks": clocks,
        "gpu_launches": K * len(calls),
        "e2e": e2e,
    }
    parity = None
    if rank == 0:
        base, parity = cpu_legs(calls, gpu_outs, world == 1 and not args.no_cpu_baseline,
                                not args.no_parity)
        if base:
            line["cpu_baseline"] = base
        # last, so that a reader of the line's tail sees them
        line["headline_kernels"] = headline_kernels(kernels)
        if parity:
            line["parity"] = parity
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    if parity and not parity["pass"]:
        raise SystemExit("parity gate failed: " + "; ".join(parity.get("failures", [])))


def step_config(world, only=None, launches=10, rank0_only=False, step_bytes=0, n_sets=1):
    """The `config` both arms print: the workload, how its inputs relate to
    the GPU's L2 (a property of the workload: both arms state it alike) and
    how it is spread."""
    cfg = dict(STEP_CONFIG) if not only else {"workload": f"subset: {only}"}
    cfg["launches_per_step"] = launches
    cfg["l2"] = (f"inputs larger than L2, no flush: steps run back to back and one step touches "
                 f"{step_bytes / 1e6:.0f} MB over {n_sets} buffer set(s), over 3x a GB300's "
                 f"L2, so every input is read from HBM")
    cfg["parallelism"] = f"rank 0 of {world}" if rank0_only and world > 1 else f"replicas x{world}"
    return cfg


def run_isolated(calls, dev, l2, peak, launches):
    """Each kernel alone: `per_graph` launches over rotating buffer sets (at
    least 3x L2 between two uses of a set) captured in one CUDA graph and
    replayed until about `launches` launches ran.  In this steady state a
    launch pays for exactly its own traffic, including the write-back of its
    own previous outputs.  ms per call = region time / launches; the median,
    min and p90 are over the per-call times of the single replays."""
    stream = torch.cuda.current_stream(dev)
    out = []
    for c in calls:
        n_sets = max(2, -(-3 * l2 // c.bytes))
        per_graph = max(20, 2 * n_sets)
        reps = max(10, -(-launches // per_graph))
        sets = device_sets([c], dev, n_sets)
        g = capture(lambda: [c.run(sets[s % n_sets][0][0], sets[s % n_sets][1][0])
                             for s in range(per_graph)], dev)
        for _ in range(3):  # warm-up: clocks and caches settle before timing
            g.replay()
        # an event between replays: the per-call time of every replay gives
        # the spread (median, min, p90) besides the overall mean
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for r in range(reps):
            g.replay()
            ev[r + 1].record(stream)
        torch.cuda.synchronize(dev)
        n = reps * per_graph
        per = sorted(ev[r].elapsed_time(ev[r + 1]) / per_graph for r in range(reps))
        ms = ev[0].elapsed_time(ev[reps]) / n
        gbs = c.bytes / (ms / 1e3) / 1e9
        out.append({"kernel": c.name, "workload": c.workload, "bytes": c.bytes,
                    "ms_per_call": round(ms, 5), "gbs": round(gbs, 1),
                    "frac_of_measured": round(gbs / peak, 4),
                    "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                    "ms_per_call_median": round(statistics.median(per), 5),
                    "ms_per_call_min": round(per[0], 5),
                    "ms_per_call_p90": round(per[min(reps - 1, int(0.9 * reps))], 5),
                    "replays": reps, "buffer_sets": n_sets, "launches": n})
        del g, sets
    return out


def gelu_rows_sweep(dev, l2, peak, launches):
    """bias_gelu_tanh fp32 at width 768 from 1k to 256k rows: device time
    per call when launches are graph-replayed back to back, and when each
    call is launched eagerly from Python, which shows where the host launch
    path, not HBM, sets the pace."""
    import window_gather_swin_gb300 as wgs
    calls = []
    for k in range(9):
        rows = 1024 << k
        x, b = synth.gelu_input(rows, 768, torch.float32, seed=4)
        calls.append(Call("bias_gelu_tanh", f"fp32 [{rows},768]", 8 * rows * 768 + 4 * 768,
                          {"x": x, "bias": b}, {"y": ((rows, 768), torch.float32)},
                          lambda i, o: wgs.bias_gelu_tanh(i["x"], i["bias"], out=o["y"]),
                          None, rows))
    graphed = run_isolated(calls, dev, l2, peak, launches)
    stream = torch.cuda.current_stream(dev)
    out = []
    for c, gr in zip(calls, graphed):
        n_sets = gr["buffer_sets"]
        sets = device_sets([c], dev, n_sets)
        n = max(50, 2 * n_sets)
        for s in range(3):
            c.run(sets[s % n_sets][0][0], sets[s % n_sets][1][0])
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for s in range(n):
            c.run(sets[s % n_sets][0][0], sets[s % n_sets][1][0])
        e.record(stream)
        torch.cuda.synchronize(dev)
        out.append({"rows": c.rows, "bytes": c.bytes, "ms_per_call": gr["ms_per_call"],
                    "gbs": gr["gbs"], "frac_of_measured": gr["frac_of_measured"],
                    "eager_ms_per_call": round(a.elapsed_time(e) / n, 5)})
        del sets
    return out


def smi_id(dev):
    """nvidia-smi --id for a torch device: its UUID when torch reports one."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    return str(dev.index)


def run_e2e(calls, dev, args, world):
    """Same metric through the public API from pinned HOST buffers: every
    step copies each call's inputs host->device, runs it, and copies its
    outputs device->host, all inside the timed region.  Copies in, kernels
    and copies out run on three streams, so call j's kernel overlaps call
    j+1's upload and call j-1's download (the host link is full duplex);
    events keep each buffer's uses in order across steps."""
    host_in = [{k: v.pin_memory() for k, v in c.inputs.items()} for c in calls]
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in c.inputs.items()} for c in calls]
    dev_out = [{k: torch.empty(s, dtype=d, device=dev) for k, (s, d) in c.outputs.items()}
               for c in calls]
    host_out = [{k: torch.empty(s, dtype=d, pin_memory=True) for k, (s, d) in c.outputs.items()}
                for c in calls]
    h2d = sum(v.numel() * v.element_size() for d in host_in for v in d.values())
    d2h = sum(v.numel() * v.element_size() for d in host_out for v in d.values())
    main = torch.cuda.current_stream(dev)
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    n = len(calls)
    ev_in, ev_run, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
    for e in ev_run + ev_out:
        e.record(main)

    def step():
        for j, (c, hi, di, do, ho) in enumerate(zip(calls, host_in, dev_in, dev_out, host_out)):
            s_in.wait_event(ev_run[j])          # the previous step's kernel has read di
            with torch.cuda.stream(s_in):
                for k in hi:
                    di[k].copy_(hi[k], non_blocking=True)
            ev_in[j].record(s_in)
            s_run.wait_event(ev_in[j])
            s_run.wait_event(ev_out[j])         # the previous step's download has read do
            with torch.cuda.stream(s_run):
                c.run(di, do)
            ev_run[j].record(s_run)
            s_out.wait_event(ev_run[j])
            with torch.cuda.stream(s_out):
                for k in do:
                    ho[k].copy_(do[k], non_blocking=True)
            ev_out[j].record(s_out)

    def join():
        for st in (s_in, s_run, s_out):
            main.wait_stream(st)

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(max(1, min(args.warmup, 3))):
        step()
    join()
    torch.cuda.synchronize(dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    for st in (s_in, s_run, s_out):
        st.wait_stream(main)
    for _ in range(steps):
        step()
    join()
    b.record(main)
    torch.cuda.synchronize(dev)
    ms = reduce_max(a.elapsed_time(b), world, dev)
    total = reduce_sum(sum(c.bytes for c in calls) * steps, world, dev)
    # the link alone, for context: one step's uploads, then its downloads
    link = {}
    for name, pairs in (("h2d_gbs", [(di[k], hi[k]) for hi, di in zip(host_in, dev_in) for k in hi]),
                        ("d2h_gbs", [(ho[k], do[k]) for do, ho in zip(dev_out, host_out) for k in do])):
        x, y = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x.record(main)
        for dst, src in pairs:
            dst.copy_(src, non_blocking=True)
        y.record(main)
        torch.cuda.synchronize(dev)
        link[name] = round((h2d if name == "h2d_gbs" else d2h) / (x.elapsed_time(y) / 1e3) / 1e9, 1)
    return {"value": round(total / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4), "link_alone": link}


# ------------------------------------------------------- reference arm ----

def run_reference(args, rank, world):
    """The oracle on the host cores, as the reference arm: each step runs
    every call of the step through the oracle, split over all usable cores,
    on the largest leading fraction of its units that keeps the whole run
    within --ref-budget-s (all of them for short runs).  Nothing here calls
    into the CUDA library: the index maps come from the oracle's builder."""
    if world > 1:
        init_dist(world, "gloo")
        if rank != 0:
            torch.distributed.destroy_process_group()
            return
    calls = build_calls(gpu=False)
    cores, model = host_cpu()
    # one whole step, untimed, sizes the sample (a small probe would be
    # dominated by the per-call cost of the thread pool)
    full_step_s, _, _ = oracle_step(calls, cores, 1.0)
    frac = args.ref_budget_s / (full_step_s * (args.steps + args.warmup))
    frac = max(1.0 / 16384, min(1.0, frac))
    for _ in range(args.warmup):
        oracle_step(calls, cores, frac)
    secs = nbytes = 0.0
    for _ in range(args.steps):
        s_, b_, _ = oracle_step(calls, cores, frac)
        secs += s_
        nbytes += b_
    value = nbytes / secs / 1e9
    sample = (f"first {frac:.3g} of the units of each of the {len(calls)} calls per step "
              f"({nbytes / args.steps / 1e6:.2f} MB algorithmic per step), split over {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded N(0,1)-family tensors of the stage shapes)",
        "config": step_config(world, None, len(calls), rank0_only=True,
                              step_bytes=sum(c.bytes for c in calls)),
        "timing": ("each step runs the oracle on every call of the step (see cpu_baseline.sample); "
                   "time.perf_counter around each call"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "sample_fraction": frac, "host_cores": cores,
                         "cpu_model": model},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1, help="ranks (one GPU each) of the run")
    p.add_argument("--steps", type=int, default=2000, help="timed steps")
    p.add_argument("--warmup", type=int, default=5, help="untimed steps before the timed ones")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours",
                   help="ours: the CUDA library; reference: the CPU oracle on a row sample")
    p.add_argument("--e2e-steps", type=int, default=20,
                   help="steps of the end-to-end leg from pinned host memory (at most --steps)")
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip timing the oracle on the host cores")
    p.add_argument("--no-parity", action="store_true",
                   help="skip the parity gate (the timed outputs against the oracle)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--ref-budget-s", type=float, default=120.0,
                   help="--impl reference: seconds of oracle work to aim for over the whole run")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the GELU rows sweep (1k-256k rows at width 768)")
    p.add_argument("--no-attribution", action="store_true",
                   help="skip the eager per-launch attribution of the step")
    p.add_argument("--isolated-launches", type=int, default=200,
                   help="launches per kernel when each kernel is timed alone")
    p.add_argument("--only", default=None,
                   help="time only the calls whose label contains this text, or equals it "
                        "when it starts with '=' (profiling aid)")
    args = p.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        p.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            p.error(f"--gpus {args.gpus} needs torchrun with {args.gpus} processes")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
