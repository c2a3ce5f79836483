"""Benchmark of the FP8 delayed-scaling linear layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic input.
The default workload is the LayerNormMLP block (16384 tokens, 4096 -> 16384 ->
4096, HYBRID delayed scaling, history 16): LayerNorm+cast, the weight casts,
fc1, GELU+cast, fc2, the grad_output cast with bias gradient, dgrad and wgrad
of both GEMMs, dGELU+cast with bias gradient, the LayerNorm backward, and one
delayed scale update of all six slots.  The default run then measures the te.Linear layer
(2048 tokens, 768 -> 3072) and the MXFP8 MLP (16384 tokens, 8192 -> 28672 -> 8192) the same
way, as the `te_linear` and `mx_mlp` entries of the same line.  `--workload NAME` runs one
workload alone (ln_mlp, llama_proj, mx_mlp, linear_hybrid, linear_fwd, ...).  Inputs are
resident in HBM before timing; the L2 is flushed (a 512 MB write) between timed steps, outside
the step events.

Prints one JSON line (rank 0).  `value` is TFLOP/s of algorithmic GEMM work
(2*M*N*K per GEMM) over the step time; `roofline` is the dominant kernel (the
GEMM) against the dense FP8 peak derived from the measured bf16 peak.
`--impl reference` times the CPU oracle (the reference arm: a plain CPU implementation
of the same computation) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "FP8 linear fwd+bwd TFLOP/s & cast/amax GB/s, % of GB300 FP8/HBM peak"
FP8_PER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor rate (4.5 : 2.25 PFLOP/s)
# DRAM bytes (read + write) per GEMM launch, the mean over one step's GEMM launches, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum of every GEMM launch of the
# workload's steps).  Each figure carries the SHA-256 of the code of the kernel sources it was
# taken with (comments left out); once that code differs, the line reports null instead.
_COMMON_SRC = ("fp8_delayed_scaling_gb300/csrc/tc.cuh", "fp8_delayed_scaling_gb300/csrc/common.cuh")
GEMM_TRAFFIC = {
    "ln_mlp": {"bytes": 1.185e9, "sources": ("fp8_delayed_scaling_gb300/csrc/gemm.cu",) + _COMMON_SRC,
               "src_sha256": "268867d7440e6b7698e6b92d11d45119dcd9845a3303220d8b49a29031b5d2c9",
               "capture": "fp8_gemm_pair_kernel<0,0,256>/<1,0,256>/<2,1,256> of commit b64b0d7, mean of the 6 "
                          "launches of a step over 17 steps"},
    # gemm.cu holds the tile order and K order the MXFP8 GEMM's host code picks
    "mx_mlp": {"bytes": 3.405e9, "sources": ("fp8_delayed_scaling_gb300/csrc/mxfp8.cu",
                                             "fp8_delayed_scaling_gb300/csrc/gemm.cu") + _COMMON_SRC,
               "src_sha256": "57296a13eb8d09eebf5e08a1917b0dd222ade21650717dfbf20ae24d43cfc7b3",
               "capture": "mxfp8_gemm_kernel of commit b64b0d7, mean of the 6 launches of a step over 17 steps"},
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def source_code(src):
    """C/C++ source without its comments and blank lines (what the compiler sees of it, near enough
    that a comment-only edit leaves it unchanged)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def source_sha(paths):
    """SHA-256 of the code of the given sources, comments left out."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel)) as f:
            h.update(source_code(f.read()).encode())
    return h.hexdigest()


def gemm_traffic(workload):
    """(bytes per launch or None, note) for the workload's GEMM launches."""
    t = GEMM_TRAFFIC.get(workload)
    if t is None:
        return None, "no capture for this workload"
    if t["src_sha256"] != source_sha(t["sources"]):
        return None, "the GEMM kernels changed since the capture"
    return t["bytes"], "ncu capture: " + t["capture"]


def measure_fp8_peak(dev, reps=10):
    """Dense FP8 library peak on this GPU: cuBLASLt E4M3 x E4M3 -> bf16 through
    torch._scaled_mm, best of `reps` launches at 8192^3 and at 16384 x 16384 x 4096, after
    ~0.3 s of back-to-back calls per shape.  Returns ({shape: TFLOP/s}, error or None)."""
    out = {}
    try:
        for M, N, K in ((8192, 8192, 8192), (16384, 16384, 4096)):
            g = torch.Generator(device="cpu").manual_seed(M + N + K)
            a = torch.randn((M, K), generator=g).mul_(0.5).to(dev).to(torch.float8_e4m3fn)
            b = torch.randn((N, K), generator=g).mul_(0.5).to(dev).to(torch.float8_e4m3fn)
            one = torch.ones((), dtype=torch.float32, device=dev)

            def f():
                return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            f()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 0.3:
                for _ in range(20):
                    f()
                torch.cuda.synchronize()
            best = float("inf")
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                f()
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1))
            out["%dx%dx%d" % (M, N, K)] = round(2.0 * M * N * K / (best * 1e-3) / 1e12, 1)
            del a, b
        return out, None
    except Exception as e:  # a library without FP8 support for this device: the derived peak stands
        return out, "%s: %s" % (type(e).__name__, str(e).splitlines()[0] if str(e) else "")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def llama_layers():
    return [(name, k, n) for name, k, n in wl.LLAMA_PROJ]


WORKLOADS = {
    "llama_proj": dict(desc="Llama-7B-shaped projections fwd+dgrad+wgrad, HYBRID delayed scaling, history 1024: "
                            "8192 tokens; QKV 4096->12288, out 4096->4096, up 4096->11008, down 11008->4096",
                       tokens=8192, layers=llama_layers(), hist=1024, fmt="hybrid", x_dtype=torch.bfloat16,
                       training=True),
    "llama_proj_mb4": dict(desc="llama_proj as 4 micro-batches of 2048 tokens with the FP8 weight cache: the weights "
                                "are cast on the first micro-batch only; scale update after every micro-batch",
                           tokens=8192, layers=llama_layers(), hist=1024, fmt="hybrid", x_dtype=torch.bfloat16,
                           training=True, micro_batches=4, weight_cache=True),
    "llama_proj_mb4_nocache": dict(desc="llama_proj_mb4 without the weight cache: every micro-batch casts the weights",
                                   tokens=8192, layers=llama_layers(), hist=1024, fmt="hybrid",
                                   x_dtype=torch.bfloat16, training=True, micro_batches=4, weight_cache=False),
    "llama_proj_current": dict(desc="llama_proj with just-in-time (current) scaling: every cast is an amax pass, the "
                                    "scale from that amax, then the cast (no history)",
                               tokens=8192, layers=llama_layers(), hist=1, fmt="hybrid", x_dtype=torch.bfloat16,
                               training=True, scaling="current"),
    "linear_hybrid": dict(desc="te.Linear 2048 tokens 768->3072 fwd+bwd, HYBRID, history 16",
                          tokens=2048, layers=[("linear", 768, 3072)], hist=16, fmt="hybrid",
                          x_dtype=torch.float32, training=True),
    "ln_mlp": dict(desc="LayerNormMLP fwd+bwd under HYBRID delayed scaling, history 16: x bf16 [16384 x 4096], "
                        "LayerNorm -> E4M3 cast -> fc1 4096->16384 -> GELU -> E4M3 cast -> fc2 16384->4096",
                   tokens=16384, layers=[("fc1", 4096, 16384), ("fc2", 16384, 4096)], hist=16, fmt="hybrid",
                   x_dtype=torch.bfloat16, training=True, kind="lnmlp"),
    "ln_mlp_separate": dict(desc="The ln_mlp block with GELU + E4M3 cast of h as its own kernel after the fc1 GEMM "
                                 "instead of in the GEMM's epilogue",
                            tokens=16384, layers=[("fc1", 4096, 16384), ("fc2", 16384, 4096)], hist=16, fmt="hybrid",
                            x_dtype=torch.bfloat16, training=True, kind="lnmlp", gelu_epilogue="separate"),
    "ln_mlp_current": dict(desc="The ln_mlp block with just-in-time (current) scaling instead of delayed scaling: "
                                "each activation is written in bf16 with its amax, then cast in a second pass",
                           tokens=16384, layers=[("fc1", 4096, 16384), ("fc2", 16384, 4096)], hist=16, fmt="hybrid",
                           x_dtype=torch.bfloat16, training=True, kind="lnmlp", scaling="current"),
    "mx_mlp": dict(desc="MXFP8 (1x32 E8M0 blocks) MLP fwd+bwd: 16384 tokens, 8192 -> 28672 -> 8192 with zero biases, "
                        "X with per-channel factors log-uniform in [1e-3, 1e2]", tokens=16384, layers=[("up", 8192, 28672),
                                                                                ("down", 28672, 8192)],
                   hist=0, fmt="mxfp8", x_dtype=torch.bfloat16, training=True, kind="mx"),
    "linear_fwd": dict(desc="te.Linear 2048 tokens 768->3072 forward, E4M3, history 16",
                       tokens=2048, layers=[("linear", 768, 3072)], hist=16, fmt="e4m3", x_dtype=torch.float32,
                       training=False),
}


def step_flops(cfg):
    M = cfg["tokens"]
    per = sum(2 * M * n * k for _, k, n in cfg["layers"])
    return per * (3 if cfg["training"] else 1)


def hbm_bytes(cfg, fused=False):
    """Algorithmic HBM bytes of one step's HBM-bound kernels, by class (each input read once,
    each output written once):
      cast     — cast + amax (+ transposed copy, + bias gradient) and MX quantisation;
      norm_act — LayerNorm forward and backward and the GELU / dGELU casts.
    With the activations fused into the GEMM epilogues (fused: GELU + cast in fc1, dGELU + cast
    + db1 in the fc2 dgrad), those passes belong to the GEMMs."""
    M = cfg["tokens"]
    if cfg.get("kind") == "mx":  # quantise X, W, dY of each layer: read 2 B, write 2 B + 2/32 B of scales;
        # dY's quantisation also writes the bias gradient (4 B per column)
        return {"cast": sum((M * k + n * k + M * n) * (2 + 2 + 2 / 32.0) + 4 * n for _, k, n in cfg["layers"])}
    if cfg.get("kind") == "lnmlp":
        H, F = cfg["layers"][0][1], cfg["layers"][0][2]
        if cfg.get("scaling") == "current":  # amax passes first, casts of the bf16 tensors after
            cast = (M * H * (2 + 2)                          # cast of the LayerNorm output y (+T)
                    + F * H * (2 + 2 + 2) * 2                # W1, W2: amax pass, cast (+T)
                    + M * F * (2 + 2)                        # cast of g (+T)
                    + M * H * (2 + 2 + 2) + 4 * H            # dY: amax pass, cast (+T, dbias)
                    + M * F * (2 + 2) + 4 * F)               # cast of dh (+T, dbias)
            norm_act = (M * H * (2 + 2) + M * F * (2 + 2) + M * F * (2 + 2 + 2) + M * H * (2 + 2 + 2))
            return {"cast": cast, "norm_act": norm_act}
        cast = F * H * (2 + 2) * 2 + M * H * (2 + 2) + 4 * H  # W1, W2 (+T); dY (+T, dbias)
        norm_act = (M * H * (2 + 2)                            # LayerNorm + cast of x (+T)
                    + (0 if fused else M * F * (2 + 2))        # GELU + cast of h (+T)
                    + (0 if fused else M * F * (2 + 2 + 2) + 4 * F)  # dGELU + cast of (dg, h) (+T, db1)
                    + M * H * (2 + 2 + 2))                     # LayerNorm backward: read dy and x, write dx
        return {"cast": cast, "norm_act": norm_act}
    esz_x = 2 if cfg["x_dtype"] == torch.bfloat16 else 4
    w_casts = 1 if cfg.get("weight_cache") else cfg.get("micro_batches", 1)  # weight casts per step
    reads = 2 if cfg.get("scaling") == "current" else 1  # just-in-time: an amax pass before each cast
    tot = 0
    for _, k, n in cfg["layers"]:
        t = 2 if cfg["training"] else 1
        tot += M * k * esz_x * reads + M * k * t          # X -> qX (+ qX^T)
        tot += (n * k * esz_x * reads + n * k * t) * w_casts  # W -> qW (+ qW^T)
        if cfg["training"]:
            tot += M * n * 2 * reads + 2 * M * n + 4 * n  # dY bf16 -> qdY + qdY^T + dbias
    return {"cast": tot}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class CycleClock:
    """Mean SM clock between two probes on a stream (fp8dl_clock_probe): each SM's cycle-counter
    delta over the global timer's, median over the SMs seen in both probes.  Unlike nvidia-smi's
    200 ms samples it covers exactly the work enqueued between the probes."""

    def __init__(self, dev, stream):
        import fp8_delayed_scaling_gb300 as fd
        self.fd = fd
        self.n = 2 * torch.cuda.get_device_properties(dev).multi_processor_count
        self.buf = [torch.zeros(3 * self.n, dtype=torch.int64, device=dev) for _ in range(2)]
        self.stream = stream

    def mark(self, k):
        self.fd.fp8dl_clock_probe(self.buf[k], self.n, self.stream)

    def mhz(self):
        """(median MHz, SMs measured); call after both marks have completed."""
        first = [{}, {}]
        for k in range(2):
            for smid, cyc, ns in self.buf[k].view(-1, 3).cpu().tolist():
                first[k].setdefault(smid, (cyc, ns))
        v = sorted((first[1][sm][0] - first[0][sm][0]) / (first[1][sm][1] - first[0][sm][1]) * 1e3
                   for sm in first[0] if sm in first[1] and first[1][sm][1] > first[0][sm][1])
        return (round(v[len(v) // 2], 1) if v else None), len(v)


class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def count(self) -> int:
        """Complete sample lines written so far."""
        if self.proc is None:
            return 0
        self.f.flush()
        try:
            with open(self.path) as f:
                return sum(1 for line in f if len(line.split(",")) >= 9 and line.endswith("\n"))
        except OSError:
            return 0

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for name, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
# Data-parallel replicas (torchrun, N > 1): the process group whose replicas share the
# scales.  Each step ends as an fp8_autocast exit does: the recorded amaxes are MAX-reduced
# over the group (one all-reduce of n_slots floats), then the scales are updated, so every
# replica casts the next step with the same scales.
GROUP = None


def close_step(state, step_no):
    if GROUP is not None:
        from fp8_delayed_scaling_gb300.autocast import reduce_amax_
        reduce_amax_(state.buf, state.n_slots, state.stride, GROUP)
    state.update(step_no)

class LnMlpModel:
    """One LayerNormMLP block (fwd+bwd) per step."""

    def __init__(self, cfg, dev, seed):
        import fp8_delayed_scaling_gb300 as fd
        from fp8_delayed_scaling_gb300.lnmlp import Fp8LayerNormMLP, make_state
        self.fd = fd
        self.cfg = cfg
        self.recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=cfg["hist"])
        self.state = make_state(self.recipe, 1, device=dev)
        M = cfg["tokens"]
        H, F = cfg["layers"][0][1], cfg["layers"][0][2]
        gamma = (1.0 + wl.normal((H,), 0.1, wl.generator(seed, "gamma"))).to(torch.bfloat16).to(dev)
        beta = torch.zeros(H, dtype=torch.bfloat16, device=dev)
        w1 = wl.normal((F, H), 0.02, wl.generator(seed, "W1"), torch.bfloat16).to(dev)
        w2 = wl.normal((H, F), 0.02, wl.generator(seed, "W2"), torch.bfloat16).to(dev)
        b1 = torch.zeros(F, dtype=torch.bfloat16, device=dev)
        b2 = torch.zeros(H, dtype=torch.bfloat16, device=dev)
        self.current = cfg.get("scaling") == "current"
        self.blk = Fp8LayerNormMLP(self.state, 0, gamma, beta, w1, b1, w2, b2, M,
                                   scaling="current" if self.current else "delayed",
                                   fused=cfg.get("gelu_epilogue", "fused") == "fused")
        self.layers = [self.blk]
        self.x = [wl.normal((M, H), 1.0, wl.generator(seed, "x"), torch.bfloat16).to(dev)]
        self.dy = [wl.normal((M, H), 1e-3, wl.generator(seed, "dY"), torch.bfloat16).to(dev)]
        self.step_no = 0
        self.blk.forward(self.x[0], seed=True)
        self.blk.backward(self.x[0], self.dy[0], seed=True)
        if not self.current:
            close_step(self.state, self.step_no)
        self.step_no += 1

    def step(self):
        self.blk.forward(self.x[0])
        self.blk.backward(self.x[0], self.dy[0])
        if not self.current:  # current scaling keeps no history to update
            close_step(self.state, self.step_no)
        self.step_no += 1

    def output_slots(self):
        """(object, attribute) of every tensor a step produces for the host, in order."""
        b = self.blk
        return [(b, "dw1"), (b, "dw2"), (b, "db1"), (b, "db2"), (b, "dgamma"), (b, "dbeta"), (b, "dx")]

    def outputs(self):
        return [getattr(o, a) for o, a in self.output_slots()]


class MxModel:
    """MXFP8 MLP: up (8192->28672) feeding down (28672->8192), fwd+bwd per step."""

    def __init__(self, cfg, dev, seed):
        import fp8_delayed_scaling_gb300 as fd
        from fp8_delayed_scaling_gb300.mxlinear import MxLinear
        self.fd = fd
        self.cfg = cfg
        M = cfg["tokens"]
        (_, H, F), _ = cfg["layers"]
        # zero biases, as in the te.Linear example (bias=True); their gradients come from the
        # column sums fused into the quantisation of dY and dh
        self.up = MxLinear(wl.normal((F, H), 0.02, wl.generator(seed, "W1"), torch.bfloat16).to(dev),
                           torch.zeros(F, dtype=torch.bfloat16, device=dev), M)
        self.down = MxLinear(wl.normal((H, F), 0.02, wl.generator(seed, "W2"), torch.bfloat16).to(dev),
                             torch.zeros(H, dtype=torch.bfloat16, device=dev), M)
        self.layers = [self.up, self.down]
        self.x = [wl.channel_scaled_normal(M, H, wl.generator(seed, "X")).to(dev)]
        self.dy = [wl.normal((M, H), 1.0, wl.generator(seed, "dY"), torch.bfloat16).to(dev)]

        class _NoState:
            def update(self, step):
                pass
        self.state = _NoState()

    def step(self):
        h = self.up.forward(self.x[0])
        self.down.forward(h)
        dh, _, _ = self.down.backward(self.dy[0])
        self.up.backward(dh)

    def output_slots(self):
        return [(self.up, "dw"), (self.down, "dw"), (self.up, "db"), (self.down, "db"), (self.up, "dx")]

    def outputs(self):
        return [getattr(o, a) for o, a in self.output_slots()]


class Model:
    def __init__(self, cfg, dev, seed):
        import fp8_delayed_scaling_gb300 as fd
        from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
        self.fd = fd
        self.cfg = cfg
        fmt = fd.FORMAT_HYBRID if cfg["fmt"] == "hybrid" else fd.FORMAT_E4M3
        self.recipe = fd.Recipe(margin=0, interval=1, fp8_format=fmt, amax_history_len=cfg["hist"])
        self.state = make_state(self.recipe, len(cfg["layers"]), device=dev)
        M = cfg["tokens"]
        self.mb = cfg.get("micro_batches", 1)
        self.cache = cfg.get("weight_cache", False)
        self.Mmb = M // self.mb  # tokens per micro-batch
        self.layers, self.x, self.dy = [], [], []
        for i, (name, k, n) in enumerate(cfg["layers"]):
            w = wl.normal((n, k), 0.02, wl.generator(seed, "W/" + name), cfg["x_dtype"]).to(dev)
            b = torch.zeros(n, dtype=cfg["x_dtype"], device=dev)
            self.layers.append(Fp8Linear(self.state, i, w, b, self.Mmb, training=cfg["training"],
                                         scaling=cfg.get("scaling", "delayed")))
            if cfg["x_dtype"] == torch.bfloat16:
                x = wl.student_t3((M, k), 0.5, wl.generator(seed, "X/" + name))
            else:
                x = wl.normal((M, k), 1.0, wl.generator(seed, "X/" + name))
            self.x.append(x.to(dev))
            if cfg["training"]:
                self.dy.append(wl.normal((M, n), 1e-3, wl.generator(seed, "dY/" + name), torch.bfloat16).to(dev))
        self.step_no = 0
        self.current = cfg.get("scaling") == "current"
        if not self.current:  # delayed scaling: the first step's amaxes seed the histories
            for lin, x in zip(self.layers, self.x):
                lin.seed_forward(x[:self.Mmb])
            for lin, dy in zip(self.layers, self.dy):
                lin.seed_backward(dy[:self.Mmb])

    def output_slots(self):
        out = []
        for lin in self.layers:
            if self.cfg["training"]:
                out += [(lin, "dw")] + ([(lin, "db")] if lin.db is not None else [])
            else:
                out.append((lin, "y"))
        return out

    def outputs(self):
        return [getattr(o, a) for o, a in self.output_slots()]

    def step(self, timers=None):
        m = self.Mmb
        for j in range(self.mb):  # one scale update per micro-batch, as at each autocast exit
            first = (j == 0) if self.cache else None
            for lin, x in zip(self.layers, self.x):
                lin.forward(x[j * m:(j + 1) * m], is_first_microbatch=first)
            for lin, dy in zip(self.layers, self.dy):
                lin.backward(dy[j * m:(j + 1) * m])
            if not self.current:  # current scaling keeps no history to update
                close_step(self.state, self.step_no)
            self.step_no += 1


def run_ours(args, cfg, dev, rank, world):
    seed = wl.SEEDS.get(args.workload, 2)
    model = {"lnmlp": LnMlpModel, "mx": MxModel}.get(cfg.get("kind"), Model)(cfg, dev, seed)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        model.step()
    torch.cuda.synchronize()

    # Single-GPU runs replay the step from a CUDA graph (StepGraph: the same launches without
    # the per-launch host cost, which decides the small layers' step time).  Their per-kernel
    # times come from eager steps directly after the timed ones (events recorded inside the
    # graph would add a dependency node between every two kernels and slow the steps they
    # time).  Several ranks (or --no-graph) step eagerly and time the kernels of the timed
    # steps themselves.  Every recipe here has interval 1, so one graph serves every step.
    use_graph = world == 1 and not args.no_graph
    timer = KernelTimer(model)
    run_step = model.step
    if use_graph:
        from fp8_delayed_scaling_gb300.graph import StepGraph
        graph = StepGraph(lambda n: model.step(), interval=1, warmup=1)
        run_step = graph.replay

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    cyc = CycleClock(dev, stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    cyc.mark(0)
    evs = []
    if not use_graph:
        timer.__enter__()
    for _ in range(args.steps):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_step()
        b.record(stream)
        evs.append((a, b))
        if not use_graph:
            torch.cuda.synchronize()  # between steps, outside the step's events
            timer.harvest()
    cyc.mark(1)
    if use_graph:
        torch.cuda.synchronize()
        # per-kernel timing pass: 5 eager steps directly after the timed steps, with no host
        # pause between, so the kernels run in the same (power-capped) state
        with timer:
            for _ in range(5):
                flush.fill_(1)
                model.step()
                torch.cuda.synchronize()
                timer.harvest()
        kt = timer.summary(timer.launches // 5)
        kt["timing"] = "events around every call of 5 eager steps right after the timed (graph-replayed) steps"
        kt["launch"] = "cuda graph per step"
    else:
        timer.__exit__(None, None, None)
        kt = timer.summary(timer.launches // args.steps)
        kt["timing"] = "events around every call of the timed steps"
        kt["launch"] = "eager, one launch at a time"
    # A timed region shorter than nvidia-smi's first samples (the small layers) is followed by
    # untimed steps of the same workload until a few samples exist (at most 3 s).  With several
    # ranks every step ends in a collective, so the ranks agree on each round (MAX of their needs).
    extra, t_extra = 0, time.perf_counter()
    while True:
        need = clocks.proc is not None and clocks.count() < 3 and time.perf_counter() - t_extra < 3.0
        if world > 1:
            flag = torch.tensor([1.0 if need else 0.0], device=dev)
            torch.distributed.all_reduce(flag, op=torch.distributed.ReduceOp.MAX)
            need = flag.item() > 0
        if not need:
            break
        for _ in range(20):
            run_step()
        extra += 20
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if clk is not None and extra:
        clk["note"] = "sampled during the timed steps and %d untimed steps of the same workload after them" % extra
    mhz, n_sm = cyc.mhz()
    if mhz is not None:
        clk = clk or {}
        clk["sm_mhz_cycles"] = mhz
        clk["sm_mhz_cycles_src"] = ("mean SM clock over the timed steps (and the L2 flushes between them): per-SM "
                                    "cycle counter over the global timer, median of %d SMs" % n_sm)
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = t.item()

    e2e = run_e2e(args, model, dev, stream, world)
    return model, ms, kt, clk, e2e


class KernelTimer:
    """CUDA events around every ABI entry point a step calls (and the scale update), by launch
    class, recorded on the stream each call is enqueued on.  After each step run inside the
    `with` block has completed, harvest() adds that step's per-call times; summary() averages
    over the harvested steps.  The library's own launch counter, read around the `with`
    block, gives the kernels enqueued in it."""
    classes = {"gemm": ["fp8_gemm", "mxfp8_gemm", "fp8_gemm_gelu_cast", "fp8_gemm_dgelu_cast"],
               "cast": ["fp8_cast_amax_transpose", "fp8_cast_amax_transpose_multi", "mxfp8_quantize"],
               "norm_act": ["fp8_layernorm_cast", "fp8_gelu_cast", "fp8_dgelu_cast", "fp8_layernorm_bwd"],
               "update": ["fp8_seed_amax_history"]}  # the just-in-time scale computation

    def __init__(self, model):
        self.model = model
        self.calls = []  # (class, entry point, start, end) of the step(s) recorded since the last harvest
        self.tot = {k: 0.0 for k in ("gemm", "cast", "norm_act", "update")}
        self.ncalls = {k: 0 for k in self.tot}
        self.by_entry = {}  # entry point -> [total ms, calls]
        self.by_call = None  # [entry point, total ms] in call order
        self.steps = 0
        self.launches = 0

    def _timed(self, kind, fn, name):
        def w(*a, **k):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(*a, **k)
            e1.record()
            self.calls.append((kind, name, e0, e1))
        return w

    def __enter__(self):
        import fp8_delayed_scaling_gb300.linear as L
        import fp8_delayed_scaling_gb300.lnmlp as LM
        import fp8_delayed_scaling_gb300.mxlinear as MX
        kind_of = {name: k for k, names in self.classes.items() for name in names}
        self.saved = [(mod, name, getattr(mod, name)) for mod in (L, LM, MX) for name in kind_of if hasattr(mod, name)]
        for mod, name, fn in self.saved:
            setattr(mod, name, self._timed(kind_of[name], fn, name))
        self.orig_update = self.model.state.update
        self.model.state.update = self._timed("update", self.orig_update, "fp8_update_scale")
        self.n0 = sys.modules["fp8_delayed_scaling_gb300"].fp8dl_kernel_launches()
        return self

    def __exit__(self, *exc):
        self.launches += sys.modules["fp8_delayed_scaling_gb300"].fp8dl_kernel_launches() - self.n0
        for mod, name, fn in self.saved:
            setattr(mod, name, fn)
        self.model.state.update = self.orig_update
        return False

    def harvest(self):
        """Add the per-call times of the step that just completed (the caller synchronised)."""
        if self.by_call is None:
            self.by_call = [[name, 0.0] for _, name, _, _ in self.calls]
        assert len(self.by_call) == len(self.calls), "every step must make the same calls"
        for i, (kind, name, e0, e1) in enumerate(self.calls):
            t = e0.elapsed_time(e1)
            self.tot[kind] += t
            self.ncalls[kind] += 1
            ent = self.by_entry.setdefault(name, [0.0, 0])
            ent[0] += t
            ent[1] += 1
            self.by_call[i][1] += t
        self.steps += 1
        self.calls = []

    def summary(self, launches_per_step):
        n = max(1, self.steps)
        out = {k: {"ms_per_step": self.tot[k] / n, "launches_per_step": self.ncalls[k] // n,
                   "avg_launch_ms": self.tot[k] / max(1, self.ncalls[k])} for k in self.tot}
        out["by_entry"] = {k: {"ms_per_step": round(v[0] / n, 5), "calls_per_step": v[1] // n}
                           for k, v in self.by_entry.items()}
        out["by_call"] = [[name, round(t / n, 5)] for name, t in (self.by_call or [])]
        model = self.model
        out["gemm"]["flops_per_step"] = step_flops(model.cfg)
        fused = getattr(getattr(model, "blk", None), "fused", False) and not getattr(model, "current", False)
        for k, v in hbm_bytes(model.cfg, fused=fused).items():
            out[k]["bytes_per_step"] = v
        if not self.ncalls["norm_act"]:
            del out["norm_act"]
        out["launches_per_step"] = launches_per_step  # the library's own kernels, counted by the library
        return out


def run_e2e(args, model, dev, stream, world):
    """Same step through the C ABI with HOST inputs and outputs: every step copies every
    layer's X and dY from pinned memory to the device and the step's products (weight and
    bias gradients, dx, ...) back to pinned memory.  The copies run through
    HostStepPipeline: on two copy streams, overlapped with the neighbouring steps' compute,
    with two input and two output sets (each step writes its products straight into the
    output set whose host copy finished, so nothing is copied on the device).  On one GPU
    the step itself is replayed from a CUDA graph captured for each pair of sets."""
    from fp8_delayed_scaling_gb300.pipeline import HostStepPipeline
    nx = len(model.x)
    host_in = [x.cpu().pin_memory() for x in model.x] + [d.cpu().pin_memory() for d in model.dy]
    slots = model.output_slots()
    dev_out = model.outputs()
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(h.numel() * h.element_size() for h in host_out)
    pipe = HostStepPipeline(model.x + model.dy, dev_out, out_sets=True)

    def eager(ins, outs):
        model.x[:] = ins[:nx]
        model.dy[:] = ins[nx:]
        for (obj, attr), t in zip(slots, outs):
            setattr(obj, attr, t)
        model.step()

    step = eager
    if world == 1 and not args.no_graph:  # one captured step per input/output set pair
        from fp8_delayed_scaling_gb300.graph import StepGraph
        graphs = []
        for k in range(2):
            ins, outs = pipe.sets[k], pipe.out_sets[k]
            graphs.append(StepGraph(lambda n, ins=ins, outs=outs: eager(ins, outs), interval=1, warmup=1))

        def step(ins, outs):
            graphs[0 if ins is pipe.sets[0] else 1].replay()

    steps = max(1, min(args.steps, 20))
    pipe.run(2, step, lambda i: host_in, lambda i: host_out)  # settle the streams and buffers
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pipe.run(steps, step, lambda i: host_in, lambda i: host_out)
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / steps
    if world > 1:
        t = torch.tensor([sec], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        sec = t.item()
    return sec, h2d, d2h


# ---------------------------------------------------------------------------
# oracle (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def run_oracle_sample(cfg, seed, rows=64, gemm_rows=8, gemm_cols=None):
    """Time the oracle on a bounded sample of one step; returns (TFLOP/s-equivalent, cores, sample text,
    estimated seconds for the whole step).

    The sample follows the workload's kind.  Per layer: the casts (per-tensor: amax + quantise;
    MX: row- and column-wise block quantisation) of `rows`-row slabs of X, W and dY, and the
    GEMM reference (per-tensor or block-scaled) of `gemm_rows` output rows (their first
    `gemm_cols` columns, all by default).  The LayerNormMLP
    adds the LayerNorm forward and backward, GELU and dGELU references on slabs.  Each part is
    scaled to the whole step by its own work (elements for element-wise parts, FLOPs for
    GEMMs), and the parts are summed."""
    import oracle
    cores = os.cpu_count() or 1
    M = cfg["tokens"]
    kind = cfg.get("kind")
    est = 0.0
    flops_done = 0
    elem_done = 0

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    def elementwise(fn, sampled, total):
        nonlocal est, elem_done
        est += timed(fn) * total / max(1, sampled)
        elem_done += sampled

    rng = np.random.default_rng(0)
    if kind == "mx":  # column-wise blocks need whole 32-row groups
        rows = max(32, rows // 32 * 32)
    for name, k, n in cfg["layers"]:
        gx = wl.generator(seed, "X/" + name)
        x = (wl.student_t3((rows, k), 0.5, gx) if cfg["x_dtype"] == torch.bfloat16
             else wl.normal((rows, k), 1.0, gx))
        w = wl.normal((rows, k), 0.02, wl.generator(seed, "W/" + name), cfg["x_dtype"])
        dy = wl.normal((rows, n), 1e-3, wl.generator(seed, "dY/" + name), torch.bfloat16)
        xa, wa, dya = wl.host_array(x), wl.host_array(w), wl.bf16_bits(dy)
        parts = [(xa, M * k), (wa, n * k)] + ([(dya, M * n)] if cfg["training"] else [])
        for arr, total in parts:
            if kind == "mx":
                elementwise(lambda: (oracle.mx_quantize_rows(arr), oracle.mx_quantize_cols(arr)), arr.size, total)
            else:
                elementwise(lambda: oracle.quantize(0, arr, float(448.0 / max(float(oracle.amax(arr)), 1e-30))),
                            arr.size, total)
        # GEMM reference: gemm_rows output rows with the full K reduction, scaled by FLOPs
        nc = n if gemm_cols is None else min(n, gemm_cols)

        def codes(r, c):  # finite E4M3 codes (0x00-0x7D), only the B rows the sample reads
            return (np.frombuffer(rng.bytes(r * c), np.uint8) % 0x7E).reshape(r, c).astype(np.uint8)

        A, B = codes(gemm_rows, k), codes(nc, k)
        ms, ns = np.meshgrid(np.arange(gemm_rows), np.arange(nc), indexing="ij")
        if kind == "mx":
            As = rng.integers(120, 134, (gemm_rows, k // 32), dtype=np.uint8)
            Bs = rng.integers(120, 134, (nc, k // 32), dtype=np.uint8)
            t = timed(lambda: oracle.mx_gemm_elems(A, As, B, Bs, None, ms.ravel(), ns.ravel()))
        else:
            t = timed(lambda: oracle.gemm_elems(A, 0, B, 0, 1.0, 1.0, None, ms.ravel(), ns.ravel()))
        flops = 2 * gemm_rows * nc * k
        est += t * (2 * M * n * k * (3 if cfg["training"] else 1)) / flops
        flops_done += flops
    if kind == "lnmlp":  # the LayerNorm and activation references on slabs
        H, F = cfg["layers"][0][1], cfg["layers"][0][2]
        g = wl.generator(seed, "lnmlp-sample")
        xs = wl.bf16_bits(wl.normal((rows, H), 1.0, g, torch.bfloat16))
        hs = wl.bf16_bits(wl.normal((rows, F), 1.0, g, torch.bfloat16))
        dgs = wl.bf16_bits(wl.normal((rows, F), 1e-3, g, torch.bfloat16))
        dys = wl.bf16_bits(wl.normal((rows, H), 1e-3, g, torch.bfloat16))
        gam = wl.bf16_bits(torch.ones(H, dtype=torch.bfloat16))
        bet = wl.bf16_bits(torch.zeros(H, dtype=torch.bfloat16))
        stats = {}
        elementwise(lambda: stats.update(fwd=oracle.layernorm_fwd(xs, gam, bet, 1e-5)), xs.size, M * H)
        elementwise(lambda: oracle.gelu(hs), hs.size, M * F)
        elementwise(lambda: oracle.dgelu(dgs, hs), hs.size, M * F)
        _, mu, rs = stats["fwd"]
        elementwise(lambda: oracle.layernorm_bwd(dys, xs, gam, mu, rs), xs.size, M * H)
    total_flops = step_flops(cfg)
    what = {"mx": "MX block quantisation (rows and columns) and the block-scaled GEMM reference",
            "lnmlp": "casts, LayerNorm fwd/bwd, GELU and dGELU references and the GEMM reference"}.get(
                kind, "casts (amax + quantise) and the GEMM reference")
    sample = ("oracle on %d host threads: %s; %d-row slabs, %d output rows per GEMM%s (%.1f MFLOP, %.2f M "
              "elements), each part scaled to one step by its elements or FLOPs"
              % (cores, what, rows, gemm_rows, "" if gemm_cols is None else " (first %d columns)" % gemm_cols,
                 flops_done / 1e6, elem_done / 1e6))
    return total_flops / est / 1e12, cores, sample, est


# ---------------------------------------------------------------------------
# single-kernel mode (for per-kernel timing and small ncu captures)
# ---------------------------------------------------------------------------
def run_only(args, dev):
    """Time one kernel alone at one shape: `--only gemm --shape M,N,K` (E4M3 x E4M3 -> bf16),
    `--only cast --shape R,C` (bf16 -> E4M3 + transposed copy + amax; `castdb`: E5M2 and the
    bias gradient, as for grad_output),
    `--only mxq --shape R,C` (bf16 -> row- and column-wise MXFP8),
    `--only mxgemm --shape M,N,K`.  Inputs are seeded; L2 is flushed between launches."""
    import fp8_delayed_scaling_gb300 as fd
    shape = [int(v) for v in args.shape.split(",")]
    g = torch.Generator(device="cpu").manual_seed(1)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    if args.only in ("gemm", "gemm_gelu", "gemm_dgelu", "mxgemm"):
        M, N, K = shape
        A = torch.randint(0, 0x70, (M, K), dtype=torch.uint8, generator=g).to(dev)
        B = torch.randint(0, 0x70, (N, K), dtype=torch.uint8, generator=g).to(dev)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        one = torch.ones(1, dtype=torch.float32, device=dev)
        if args.only == "gemm":
            fn = lambda: fd.fp8_gemm(A, fd.E4M3, B, fd.E4M3, one, one, D)  # noqa: E731
        elif args.only == "gemm_gelu":
            q = torch.empty((M, N), dtype=torch.uint8, device=dev)
            qt = torch.empty((N, M), dtype=torch.uint8, device=dev)
            am = torch.zeros(1, dtype=torch.float32, device=dev)
            fn = lambda: fd.fp8_gemm_gelu_cast(A, fd.E4M3, B, fd.E4M3, one, one, D, fd.E4M3, one, q, qt,  # noqa: E731
                                               q_amax=am)
        elif args.only == "gemm_dgelu":
            h = wl.normal((M, N), 2.0, g, torch.bfloat16).to(dev)
            q = torch.empty((M, N), dtype=torch.uint8, device=dev)
            qt = torch.empty((N, M), dtype=torch.uint8, device=dev)
            am = torch.zeros(1, dtype=torch.float32, device=dev)
            db = torch.empty(N, dtype=torch.float32, device=dev)
            ws = torch.empty(fd.fp8_gemm_dgelu_workspace_size(M, N), dtype=torch.uint8, device=dev)
            fn = lambda: fd.fp8_gemm_dgelu_cast(A, fd.E5M2, B, fd.E4M3, one, one, h, fd.E5M2, one, q, qt,  # noqa: E731
                                                q_amax=am, dbias=db, workspace=ws)
        else:
            As = torch.randint(120, 134, (M, K // 32), dtype=torch.uint8, generator=g).to(dev)
            Bs = torch.randint(120, 134, (N, K // 32), dtype=torch.uint8, generator=g).to(dev)
            fn = lambda: fd.mxfp8_gemm(A, As, B, Bs, D)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif args.only in ("gelu", "dgelu", "ln", "lnbwd"):
        R, C = shape
        x = wl.normal((R, C), 2.0, g, torch.bfloat16).to(dev)
        sc = torch.ones(1, dtype=torch.float32, device=dev)
        am = torch.zeros(1, dtype=torch.float32, device=dev)
        q = torch.empty((R, C), dtype=torch.uint8, device=dev)
        qt = torch.empty((C, R), dtype=torch.uint8, device=dev)
        if args.only == "gelu":
            fn = lambda: fd.fp8_gelu_cast(x, fd.E4M3, sc, out=q, out_t=qt, amax=am)  # noqa: E731
            work = R * C * (2 + 1 + 1)
        elif args.only == "dgelu":
            dgt = wl.normal((R, C), 1e-3, g, torch.bfloat16).to(dev)
            db = torch.empty(C, dtype=torch.float32, device=dev)
            ws = torch.empty(fd.fp8_cast_workspace_size(R, C), dtype=torch.uint8, device=dev)
            fn = lambda: fd.fp8_dgelu_cast(dgt, x, fd.E5M2, sc, out=q, out_t=qt, amax=am, dbias=db,  # noqa: E731
                                           workspace=ws)
            work = R * C * (2 + 2 + 1 + 1) + 4 * C
        elif args.only == "ln":
            gam = torch.ones(C, dtype=torch.bfloat16, device=dev)
            bet = torch.zeros(C, dtype=torch.bfloat16, device=dev)
            mu = torch.empty(R, dtype=torch.float32, device=dev)
            rs = torch.empty(R, dtype=torch.float32, device=dev)
            fn = lambda: fd.fp8_layernorm_cast(x, gam, bet, 1e-5, fd.E4M3, sc, mu, rs, out=q, out_t=qt,  # noqa: E731
                                               amax=am)
            work = R * C * (2 + 1 + 1) + 8 * R
        else:
            gam = torch.ones(C, dtype=torch.bfloat16, device=dev)
            mu = torch.zeros(R, dtype=torch.float32, device=dev)
            rs = torch.ones(R, dtype=torch.float32, device=dev)
            dyt = wl.normal((R, C), 1e-3, g, torch.bfloat16).to(dev)
            dx = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
            dgm = torch.empty(C, dtype=torch.float32, device=dev)
            dbt = torch.empty(C, dtype=torch.float32, device=dev)
            ws = torch.empty(fd.fp8_layernorm_bwd_workspace_size(R, C), dtype=torch.uint8, device=dev)
            fn = lambda: fd.fp8_layernorm_bwd(dyt, x, gam, mu, rs, dx, dgm, dbt, ws)  # noqa: E731
            work = R * C * (2 + 2 + 2) + 8 * C
        unit = "GB/s"
    else:
        R, C = shape
        x = wl.normal((R, C), 1.0, g, torch.bfloat16).to(dev)
        if args.only in ("cast", "castdb"):
            q = torch.empty((R, C), dtype=torch.uint8, device=dev)
            qt = torch.empty((C, R), dtype=torch.uint8, device=dev)
            sc = torch.ones(1, dtype=torch.float32, device=dev)
            am = torch.zeros(1, dtype=torch.float32, device=dev)
            if args.only == "cast":
                fn = lambda: fd.fp8_cast_amax_transpose(x, fd.E4M3, sc, out=q, out_t=qt, amax=am)  # noqa: E731
                work = R * C * (2 + 1 + 1)
            else:  # the grad_output cast of a layer with a bias: E5M2 codes and the column sums
                db = torch.empty(C, dtype=torch.float32, device=dev)
                ws = torch.empty(fd.fp8_cast_workspace_size(R, C), dtype=torch.uint8, device=dev)
                fn = lambda: fd.fp8_cast_amax_transpose(x, fd.E5M2, sc, out=q, out_t=qt, amax=am,  # noqa: E731
                                                        dbias=db, workspace=ws)
                work = R * C * (2 + 1 + 1) + 4 * C
        else:
            rq = torch.empty((R, C), dtype=torch.uint8, device=dev)
            rs = torch.empty((R, C // 32), dtype=torch.uint8, device=dev)
            cq = torch.empty((C, R), dtype=torch.uint8, device=dev)
            cs = torch.empty((C, R // 32), dtype=torch.uint8, device=dev)
            fn = lambda: fd.mxfp8_quantize(x, rq, rs, cq, cs)  # noqa: E731
            work = R * C * (2 + 1 + 1) + 2 * R * C // 32
        unit = "GB/s"
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    avg = sum(ms) / len(ms)
    rate = work / (avg * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"only": args.only, "shape": shape, "avg_ms": round(avg, 5), "min_ms": round(min(ms), 5),
                      "rate": round(rate, 1), "unit": unit, "launches": args.warmup + args.steps}))


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None, choices=sorted(WORKLOADS),
                    help="one workload alone; without it: ln_mlp, then te.Linear and the MXFP8 MLP beside it")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", default=None, choices=["gemm", "gemm_gelu", "gemm_dgelu", "cast", "castdb", "mxq", "mxgemm", "gelu", "dgelu",
                                                          "ln", "lnbwd"])
    ap.add_argument("--shape", default="8192,12288,4096")
    ap.add_argument("--no-graph", action="store_true", help="issue the timed steps one launch at a time")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    default_run = args.workload is None
    if default_run:
        args.workload = "ln_mlp"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    # identical in both arms: how the GPU arm launches its kernels is the top-level "launch" key
    config = {"workload": args.workload, "desc": cfg["desc"], "tokens": cfg["tokens"],
              "l2": "flushed between timed steps (512 MB write)", "parallelism": "replicas" if world > 1 else "single"}

    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle as it stands on the host cores: W untimed and K timed steps, each a bounded
        # sample of the step scaled to the whole step.  The sample is the cpu_baseline one
        # (64-row slabs, 8 output rows per GEMM) unless W + K of those would take more than
        # ~150 s; then 16-row slabs and 2048 columns of one output row per GEMM.
        t0 = time.perf_counter()
        run_oracle_sample(cfg, 2)
        small = (time.perf_counter() - t0) * (args.steps + args.warmup) > 150.0
        kw = dict(rows=16, gemm_rows=1, gemm_cols=2048) if small else {}
        for _ in range(args.warmup - 1):
            run_oracle_sample(cfg, 2, **kw)
        est = []
        t_timed = time.perf_counter()
        for _ in range(args.steps):
            val, cores, sample, step_s = run_oracle_sample(cfg, 2, **kw)
            est.append(step_s)
        wall = time.perf_counter() - t_timed
        step_s = sum(est) / len(est)
        val = step_flops(cfg) / step_s / 1e12
        line = {"impl": "reference", "metric": METRIC, "value": val,
                "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": config,
                # a whole step of the oracle would take minutes: each timed step is a bounded
                # sample, and ms_per_step is that sample's time scaled to one whole step
                "extrapolated": True, "timed_wall_s": round(wall, 3),
                "sampled_ms_per_step": round(wall / args.steps * 1e3, 3),
                "launch": "host (the oracle on the CPU cores)",
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    torch.cuda.set_device(local)
    if world > 1:
        global GROUP
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
        GROUP = torch.distributed.group.WORLD
    dev = torch.device("cuda", local)
    if args.only:
        if rank == 0:
            run_only(args, dev)
        return
    # The dense FP8 denominator: the larger of the measured bf16 burst x the nominal 2:1 ratio
    # and cuBLASLt's own FP8 GEMM rate measured here, before the workload, at full clocks.
    # Both are burst figures: the bench's GEMMs run in steps of milliseconds, not in the
    # seconds-long loop the sustained (power-capped) figure comes from, which is kept beside.
    clocks_peak = ClockSampler(dev.index if dev.index is not None else 0)
    clocks_peak.start()
    scaled_mm, scaled_mm_err = measure_fp8_peak(dev)
    clk_peak = clocks_peak.stop()
    derived = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * FP8_PER_BF16
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) * FP8_PER_BF16
    lib_fp8 = max(scaled_mm.values()) if scaled_mm else 0.0
    fp8_peak = max(derived, lib_fp8)
    peak_src = ("cuBLASLt FP8 E4M3 GEMM (torch._scaled_mm) measured in this run, best of 10 at %s"
                % max(scaled_mm, key=scaled_mm.get) if lib_fp8 > derived else
                "%s bf16 burst x %.0f (nominal FP8:BF16)" % (peak_src, FP8_PER_BF16))
    fp8_peak_info = {"used": round(fp8_peak, 1), "bf16_burst_x2": round(derived, 1), "scaled_mm": scaled_mm,
                     "scaled_mm_error": scaled_mm_err, "clocks": clk_peak,
                     "sustained_bf16_x2": round(sustained, 1)}
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])

    def hbm_class(c):  # achieved GB/s of algorithmic bytes against the HBM peak
        gbs = c["bytes_per_step"] / (c["ms_per_step"] * 1e-3) / 1e9
        return {"achieved_gbs": round(gbs, 1), "peak_gbs": hbm, "frac": round(gbs / hbm, 4),
                "ms_per_step": round(c["ms_per_step"], 4), "launches_per_step": c["launches_per_step"]}

    def roofline(wcfg, wname, kt, clk):
        """The workload's dominant kernel class, its GEMMs: algorithmic FLOPs of a step's GEMM
        launches over their summed CUDA-event durations, against the burst FP8 peak.  Side keys:
        the fraction of the sustained peak, and of the burst peak scaled to the SM clock the
        cycle counters measured over the timed steps (what the same GEMMs could do at that clock)."""
        g = kt["gemm"]
        achieved = g["flops_per_step"] / (g["ms_per_step"] * 1e-3) / 1e12
        traffic, tnote = gemm_traffic(wname)
        r = {"bound": "tensor", "kernel": "mxfp8_gemm" if wcfg.get("kind") == "mx" else "fp8_gemm",
             "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
             "frac": round(achieved / fp8_peak, 4), "traffic": traffic, "traffic_src": tnote,
             "peak_src": peak_src, "gemm_ms_per_step": round(g["ms_per_step"], 4),
             "gemm_launches_per_step": g["launches_per_step"],
             "frac_of_sustained": round(achieved / sustained, 4)}
        if clk and clk.get("sm_mhz_cycles"):
            top = clk.get("sm_max_mhz") or 2070.0
            r["frac_at_clock"] = round(achieved / (fp8_peak * clk["sm_mhz_cycles"] / top), 4)
            r["frac_at_clock_src"] = "burst peak x sm_mhz_cycles / sm_max_mhz (%.0f / %.0f MHz)" % (
                clk["sm_mhz_cycles"], top)
        return r

    model, ms, kt, clk, (e2e_s, h2d, d2h) = run_ours(args, cfg, dev, rank, world)
    launch = kt.pop("launch")
    flops = step_flops(cfg)
    value = flops * world / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8(e4m3/e5m2)->fp32acc->bf16", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": config, "launch": launch,
        "roofline": roofline(cfg, args.workload, kt, clk),
        "fp8_peak": fp8_peak_info,
        "cast": hbm_class(kt["cast"]),
        "kernels": {k: ({kk: (round(vv, 5) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                        if isinstance(v, dict) else v) for k, v in kt.items() if k != "launches_per_step"},
        "gpu_launches": kt["launches_per_step"] * args.steps,
        "e2e": {"value": round(flops * world / e2e_s / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "H2D of the next step and D2H of the previous one overlap this step's compute "
                          "(two copy streams, two buffer sets)"},
    }
    if "norm_act" in kt:
        line["norm_act"] = hbm_class(kt["norm_act"])
    if clk:
        line["clocks"] = clk
    if world == 1 and default_run:
        # Two more workloads measured the same way right after the main one, so one line carries
        # them: the te.Linear layer of the pages' fwd+bwd HYBRID recipe (2048 tokens, 768 -> 3072)
        # and the MXFP8 MLP (16384 tokens, 8192 -> 28672 -> 8192), the largest configuration.
        del model
        for key, wname in (("te_linear", "linear_hybrid"), ("mx_mlp", "mx_mlp")):
            sub = argparse.Namespace(**vars(args))
            sub.workload = wname
            scfg = WORKLOADS[wname]
            smodel, s_ms, s_kt, s_clk, (s_e2e, s_h2d, s_d2h) = run_ours(sub, scfg, dev, rank, world)
            del smodel
            s_flops = step_flops(scfg)
            entry = {
                "workload": wname, "desc": scfg["desc"], "tokens": scfg["tokens"],
                "value": round(s_flops / (s_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(s_ms, 4),
                "steps": sub.steps, "launch": s_kt.pop("launch"),
                "gpu_launches": s_kt["launches_per_step"] * sub.steps,
                "e2e": {"value": round(s_flops / s_e2e / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": s_h2d,
                        "d2h_bytes_per_step": s_d2h}}
            if key == "mx_mlp":
                entry["roofline"] = roofline(scfg, wname, s_kt, s_clk)
                entry["quantize"] = hbm_class(s_kt["cast"])
                entry["by_entry"] = s_kt["by_entry"]
                if s_clk:
                    entry["clocks"] = s_clk
            line[key] = entry
            torch.cuda.empty_cache()
    if rank == 0 and world == 1:
        val, cores, sample, _ = run_oracle_sample(cfg, 2)
        line["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
