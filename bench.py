#!/usr/bin/env python
"""Benchmark of the quantized matmul hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qmm|reference]

Prints ONE JSON line (rank 0).  The headline workload is the Q4_0 x Q8_0
decode GEMV over a 7B-style layer set at m = 1 (K=4096 -> N = 4096 x4,
11008 x2; K=11008 -> N=4096): one step quantizes each matrix's f32
activation row to Q8_0 and runs the GEMV, for all seven matrices.  `value`
is whole-job HBM throughput in GB/s: the algorithmic bytes of a step times
the steps all ranks ran, divided by the slowest rank's device time.  The
other workloads (single 4096x4096 GEMV, BitNet ternary GEMV, the 512 x
14336 x 4096 prefill GEMM on the tensor cores, the 4096 -> 128256 vocabulary
projection at m = 1, 16, 128) are reported under "configs".

Timing: steps run as CUDA-graph replays (so host launch overhead does not
enter the device time), timed with CUDA events on the launching stream
after the warm-up, with a device synchronize (and a barrier under
torchrun) on both sides.  Each workload rotates through enough copies of
its weights that the bytes touched between two uses of one copy exceed
twice the 129 MB L2, so every step streams its weights from HBM.

--impl reference times the CPU oracle (tests-only scalar C) on the host
cores on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

QK = 32
L2_BYTES = 129 * 10**6
METRIC = "decode GEMV achieved HBM GB/s (% of peak); prefill GEMM int8 TOPS (% of peak)"
# the GB300's nominal HBM3e bandwidth (~8 TB/s); fractions are reported against
# it beside the measured copy peak
NOMINAL_HBM_GBS = 8000.0
LAYER_SET = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]  # (N, K), seeds 1..7
WORKLOAD_C2 = ("Q4_0xQ8_0 decode GEMV over a 7B-style layer set, m=1: K=4096 -> N in "
               "{4096 x4, 11008 x2}, K=11008 -> N=4096; weights ~N(0,0.02) seeds 1-7, "
               "activations ~N(0,1); one step = Q8_0-quantize each f32 activation row and "
               "run the GEMV, all 7 matrices as independent problems (each has its own x): "
               "qmm_linear_q4_0_grouped, one quantizer launch + one GEMV launch, PDL")


# ---------------------------------------------------------------------------
# algorithmic bytes and ops (per launch / per step)

def q4_weight_bytes(n, k):
    return n * k // 2 + 2 * n * (k // QK)


def gemv_bytes(m, n, k):
    """Q4_0 weights + Q8_0 activations (codes + scales) + f32 output."""
    return q4_weight_bytes(n, k) + m * k + 2 * m * (k // QK) + 4 * m * n


def quant_bytes(m, k):
    """f32 activations in, Q8_0 codes + fp16 scales out."""
    return 4 * m * k + m * k + 2 * m * (k // QK)


def linear_bytes(m, n, k):
    """Decode layer as a whole: Q4_0 weights + f32 activations in + f32
    output (the Q8_0 intermediate is not counted)."""
    return q4_weight_bytes(n, k) + 4 * m * k + 4 * m * n


def bitnet_bytes(m, n, k):
    """Ternary GEMV: packed codes + int8 activations, scale and sum + f32 output."""
    return n * k // 4 + m * k + 8 * m + 4 * m * n


def bitnet_step_bytes(m, n, k):
    """BitNet decode layer as a whole: packed codes + f32 activations in +
    f32 output (the int8 intermediate is not counted)."""
    return n * k // 4 + 4 * m * k + 4 * m * n


def copies_for(bytes_per_copy):
    """Rotation depth so that the other copies touched between two uses of
    one copy exceed twice the L2."""
    return max(1, -(-2 * L2_BYTES // max(1, bytes_per_copy)) + 1)


# ---------------------------------------------------------------------------
# environment helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# the layer-set step's GEMV (rows per warp, PDL, warps per CTA), as ncu names it
HEADLINE_KERNEL = "gemv_grouped_m1_staged_kernel<2,1,4>"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the last ncu capture, as recorded
    in profiles/traffic.txt (kernel, bytes, sha256 of the kernel's source
    file, that file), or None when there is no record or the source changed
    since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel:
                src = os.path.join(ROOT, parts[3])
                if not os.path.exists(src):
                    return None
                with open(src, "rb") as g:
                    digest = hashlib.sha256(g.read()).hexdigest()
                return int(parts[1]) if digest == parts[2] else None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().strip().splitlines() if r.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("nccl" if self._cuda() else "gloo")
            self.pg = dist

    @staticmethod
    def _cuda():
        import torch
        return torch.cuda.is_available()

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if self._cuda() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# timing of captured steps

class GraphTimer:
    """Captures `step(i)` for whole rotations of `rot` steps (about 32 steps)
    into a CUDA graph and times K steps as graph replays with CUDA events.
    Consecutive steps inside one graph overlap through programmatic dependent
    launch; a graph boundary does not, so larger graphs leave fewer such
    breaks per step."""

    def __init__(self, step, rot: int, unit_steps: int = 32):
        import torch
        self.torch = torch
        self.step = step
        self.rot = rot * max(1, unit_steps // rot)  # steps per full graph
        for i in range(rot):  # eager run: one-time setup inside the library
            step(i)
        torch.cuda.synchronize()
        self.full = self._capture(range(self.rot))
        self.tails = {}

    def _capture(self, idx):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in idx:
                self.step(i)
        return g

    def _tail(self, t):
        if t not in self.tails:
            self.tails[t] = self._capture(range(t))
        return self.tails[t]

    def run(self, k: int):
        for _ in range(k // self.rot):
            self.full.replay()
        if k % self.rot:
            self._tail(k % self.rot).replay()

    def median(self, k: int, warmup: int, dist: Dist, repeats: int = 3):
        """Times k steps `repeats` times (the first after `warmup` untimed
        steps) and returns the median time with the spread: CV over the
        repeats and NOISY when it passes 8%."""
        runs = [self.time(k, warmup if r == 0 else 1, dist)[0] for r in range(repeats)]
        mean = sum(runs) / len(runs)
        cv = (sum((v - mean) ** 2 for v in runs) / len(runs)) ** 0.5 / mean
        return statistics.median(runs), {"repeats": repeats, "cv": round(cv, 5),
                                         "noisy": cv > 0.08}

    def time(self, k: int, warmup: int, dist: Dist, sampler: ClockSampler | None = None,
             settle_s: float = 0.6):
        """Times exactly k steps after `warmup` untimed ones.  With a clock
        sampler, nvidia-smi samples from just before an untimed block of
        replays of about settle_s seconds (which runs right before the timed
        region) until the timed region ends, so a short timed region still
        has clock samples taken under the same load at the same moment."""
        torch = self.torch
        if k % self.rot:
            self._tail(k % self.rot)
        self.run(max(warmup, 1))
        torch.cuda.synchronize()
        settle = 0
        if sampler:
            t0 = time.perf_counter()
            self.run(self.rot)
            torch.cuda.synchronize()
            per_step = max((time.perf_counter() - t0) / self.rot, 1e-7)
            settle = int(settle_s / per_step) // self.rot * self.rot
        dist.barrier()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if sampler:
            sampler.start()
            self.run(settle)
        start.record()
        self.run(k)
        end.record()
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        if clocks is not None:
            clocks["window"] = (f"nvidia-smi every 100 ms over {settle} untimed replays of the "
                                f"same step and the {k} timed ones right after them")
        dist.barrier()
        ms = dist.max(start.elapsed_time(end))
        return ms, clocks


# ---------------------------------------------------------------------------
# workloads (GPU)

def _up(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _quantized_weights(q, seed, n, k, m, copies, **kw):
    """Draws f32 weights and activations, quantizes the weights on the GPU,
    and returns `copies` independent copies of (wq, wd) plus x."""
    from quantized_matmul_gb300 import synthetic
    w, x = synthetic.q4_0_case(seed, n, k, m, **kw)
    wdev = _up(w)
    wq, wd = q.quantize_weight_q4_0(wdev)
    del wdev
    out = [(wq, wd)] + [(wq.clone(), wd.clone()) for _ in range(copies - 1)]
    return out, x


def run_layer_set(q, args, dist, peaks):
    import torch
    set_bytes = sum(q4_weight_bytes(n, k) for n, k in LAYER_SET)
    rot = copies_for(set_bytes)
    mats = []
    for j, (n, k) in enumerate(LAYER_SET):
        wts, x = _quantized_weights(q, j + 1, n, k, 1, rot)
        xd = _up(x)
        aq = torch.empty((1, k), dtype=torch.int8, device="cuda")
        ad = torch.empty((1, k // QK), dtype=torch.float16, device="cuda")
        y = torch.empty((1, n), dtype=torch.float32, device="cuda")
        mats.append(dict(n=n, k=k, wts=wts, x=xd, aq=aq, ad=ad, y=y, x_host=x))
    torch.cuda.synchronize()

    def grouped_step(pdl):
        tables = [[(mt["x"], *mt["wts"][c], mt["y"], mt["aq"], mt["ad"]) for mt in mats]
                  for c in range(rot)]

        def step(i):
            q.linear_q4_0_grouped(tables[i % rot], pdl=pdl)
        return step

    def chain_step(pdl):
        def step(i):
            c = i % rot
            for mt in mats:
                wq, wd = mt["wts"][c]
                q.linear_q4_0(mt["x"], wq, wd, y=mt["y"], pdl=pdl, aq=mt["aq"], ad=mt["ad"])
        return step

    def two_kernel_step(i):
        c = i % rot
        for mt in mats:
            wq, wd = mt["wts"][c]
            q.quantize_act_q8_0(mt["x"], mt["aq"], mt["ad"])
            q.gemv_q4_0_q8_0(wq, wd, mt["aq"], mt["ad"], y=mt["y"], split_k=1)

    def gemv_only(i):
        c = i % rot
        for mt in mats:
            wq, wd = mt["wts"][c]
            q.gemv_q4_0_q8_0(wq, wd, mt["aq"], mt["ad"], y=mt["y"], split_k=1)

    step_bytes = sum(linear_bytes(1, n, k) for n, k in LAYER_SET)
    gemv_step_bytes = sum(gemv_bytes(1, n, k) for n, k in LAYER_SET)

    def gbs(ms_, nbytes):
        return round(nbytes * args.steps / (ms_ * 1e-3) / 1e9, 1)

    sampler = ClockSampler(torch.cuda.current_device())
    timer = GraphTimer(grouped_step(True), rot)
    ms, clocks = timer.time(args.steps, args.warmup, dist, sampler)
    value = dist.world * step_bytes * args.steps / (ms * 1e-3) / 1e9
    # run-to-run spread: five more timed regions of a fifth of the steps each
    # (outside the headline's region; they only describe its noise)
    rep_steps = max(args.steps // 5, 1)
    reps = [timer.time(rep_steps, 1, dist)[0] for _ in range(5)]
    rep_mean = sum(reps) / len(reps)
    rep_cv = (sum((r - rep_mean) ** 2 for r in reps) / len(reps)) ** 0.5 / rep_mean
    noise = {"repeats": len(reps), "steps_each": rep_steps, "cv": round(rep_cv, 5),
             "noisy": rep_cv > 0.08}
    variants = {}
    for name, fn, what in (
            ("grouped_no_pdl", grouped_step(False), "the same two launches without PDL"),
            ("chain_pdl", chain_step(True), "the 7 matrices as a dependent chain: "
             "qmm_linear_q4_0 per matrix with PDL (14 launches)"),
            ("chain_no_pdl", chain_step(False), "qmm_linear_q4_0 per matrix, no PDL"),
            ("quantize_then_gemv", two_kernel_step, "qmm_quantize_act_q8_0 + "
             "qmm_gemv_q4_0_q8_0 per matrix, plain launches")):
        ms_v, noise_v = GraphTimer(fn, rot).median(args.steps, args.warmup, dist)
        variants[name] = {"value": gbs(ms_v, step_bytes), "unit": "GB/s", "noise": noise_v,
                          "ms_per_step": round(ms_v / args.steps, 6), "path": what}
    # the step's dominant kernel is the grouped one-token GEMV (the quantizer
    # moves 0.3% of the bytes); with PDL the two launches overlap, so its
    # time is bounded by the step time, which is what is measured
    achieved = step_bytes * args.steps / (ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": HEADLINE_KERNEL,
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"],
                "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "nominal_peak": NOMINAL_HBM_GBS,
                "traffic": recorded_traffic(HEADLINE_KERNEL),
                "traffic_source": "profiles/traffic.txt (ncu dram__bytes_read.sum + "
                                  "dram__bytes_write.sum of one launch; null once the kernel's "
                                  "source changed since that capture)",
                "algorithmic_bytes_per_launch": step_bytes,
                "avg_launch_us": round(ms * 1e3 / args.steps, 3),
                "measured": "the timed step (one grouped quantizer launch + one grouped GEMV "
                            "launch, overlapped by PDL) per launch of the GEMV, CUDA events on "
                            "the replay stream"}
    # the GEMV kernel alone on pre-quantized activations, same 7 matrices
    ms_g, noise_g = GraphTimer(gemv_only, rot).median(args.steps, args.warmup, dist)
    variants["gemv_only_prequantized"] = {"noise": noise_g,
        "value": gbs(ms_g, gemv_step_bytes), "unit": "GB/s",
        "bytes": "weights + Q8_0 activations + f32 y", "ms_per_step": round(ms_g / args.steps, 6)}

    # end to end through the public API, one eager call per step: the 7
    # activation rows in one pinned host buffer go in with one copy, the
    # grouped step runs, and the 7 outputs (one device buffer) come back to
    # one pinned host buffer with one copy, all enqueued by one C-ABI call
    # (qmm_linear_q4_0_grouped_host, through GroupedLinear(host_io=...))
    k_off = [int(v) for v in np.cumsum([0] + [k for _, k in LAYER_SET])]
    n_off = [int(v) for v in np.cumsum([0] + [n for n, _ in LAYER_SET])]
    x_h = torch.from_numpy(np.concatenate([mt["x_host"].ravel() for mt in mats])).pin_memory()
    y_h = torch.empty((n_off[-1],), dtype=torch.float32).pin_memory()
    x_d = torch.empty_like(x_h, device="cuda")
    y_d = torch.empty((n_off[-1],), dtype=torch.float32, device="cuda")
    e2e_steps = max(20, min(args.steps, 400))
    calls = [q.GroupedLinear([(x_d[k_off[j]:k_off[j + 1]].view(1, -1), *mt["wts"][c],
                               y_d[n_off[j]:n_off[j + 1]].view(1, -1), mt["aq"], mt["ad"])
                              for j, mt in enumerate(mats)], pdl=True,
                             host_io=(x_h, x_d, y_d, y_h), host_direct=True)
             for c in range(rot)]

    def e2e_step(i):
        calls[i % rot]()

    direct = q.host_addressable(x_h) and q.host_addressable(y_h)
    e2e_path = ("one eager public-API call per step (GroupedLinear with host_io, host_direct -> "
                "qmm_linear_q4_0_grouped_host): " +
                ("the grouped quantizer reads the 7 activation rows from page-locked host "
                 "memory and the GEMV writes the 7 outputs to page-locked host memory, over "
                 "NVLink-C2C (the device addresses both buffers)" if direct else
                 "a pinned host->device copy of the 7 activation rows, the grouped quantizer + "
                 "GEMV (PDL), a device->host copy of the 7 outputs into pinned memory"))

    for i in range(max(3, min(args.warmup, 50))):
        e2e_step(i)
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = dist.max(time.perf_counter() - t0)
    # the same calls as a token loop must run them: each step's outputs are
    # in host memory (the stream synchronized) before the next step is issued;
    # such a loop replays the step as a CUDA graph (GroupedLinear(graph=True):
    # one launch per step), the eager form is reported beside it
    sync_steps = max(20, min(args.steps, 200))
    gcalls = [q.GroupedLinear([(x_d[k_off[j]:k_off[j + 1]].view(1, -1), *mt["wts"][c],
                                y_d[n_off[j]:n_off[j + 1]].view(1, -1), mt["aq"], mt["ad"])
                               for j, mt in enumerate(mats)], pdl=True,
                              host_io=(x_h, x_d, y_d, y_h), host_direct=True, graph=True)
              for c in range(rot)]
    for i in range(max(3, rot)):
        gcalls[i % rot]()  # first call of each: run and capture
    torch.cuda.synchronize()

    def sync_loop(fn):
        dist.barrier()
        t0 = time.perf_counter()
        for i in range(sync_steps):
            fn(i)
            torch.cuda.current_stream().synchronize()
        return dist.max(time.perf_counter() - t0)

    sync_s = sync_loop(lambda i: gcalls[i % rot]())
    sync_eager_s = sync_loop(e2e_step)
    e2e = {"value": round(dist.world * step_bytes * e2e_steps / e2e_s / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": sum(4 * k for _, k in LAYER_SET),
           "d2h_bytes_per_step": sum(4 * n for n, _ in LAYER_SET),
           "steps": e2e_steps, "path": e2e_path,
           "timing": "steps issued back to back, one synchronize at the end (pipelined)",
           "synchronized": {"value": round(dist.world * step_bytes * sync_steps / sync_s / 1e9, 2),
                            "unit": "GB/s", "us_per_step": round(sync_s * 1e6 / sync_steps, 2),
                            "steps": sync_steps,
                            "path": "GroupedLinear(..., host_direct=True, graph=True): the step "
                                    "captured once and replayed as a CUDA graph",
                            "timing": "each step's outputs in host memory (stream synchronized) "
                                      "before the next step is issued, as a token loop runs",
                            "eager": {"value": round(dist.world * step_bytes * sync_steps /
                                                     sync_eager_s / 1e9, 2),
                                      "us_per_step": round(sync_eager_s * 1e6 / sync_steps, 2),
                                      "path": "the same with one eager call per step"}}}
    return dict(value=value, ms=ms / args.steps, clocks=clocks, roofline=roofline, e2e=e2e, noise=noise,
                launches=2 * args.steps, rot=rot, set_bytes=set_bytes,
                step_bytes=step_bytes, variants=variants)


def run_single_gemv(q, steps, warmup, dist, peaks):
    import torch
    n, k = 4096, 4096
    rot = copies_for(q4_weight_bytes(n, k))
    wts, x = _quantized_weights(q, 0, n, k, 1, rot)
    aq, ad = q.quantize_act_q8_0(_up(x))
    y = torch.empty((1, n), dtype=torch.float32, device="cuda")

    def step(i):
        wq, wd = wts[i % rot]
        q.gemv_q4_0_q8_0(wq, wd, aq, ad, y=y, split_k=1)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    gbs = dist.world * gemv_bytes(1, n, k) * steps / (ms * 1e-3) / 1e9
    return {"workload": "Q4_0xQ8_0 GEMV m=1 K=4096 N=4096 (seed 0)", "value": round(gbs, 1),
            "unit": "GB/s", "frac_hbm": round(gbs / dist.world / peaks["hbm_gbs"], 4),
            "us_per_launch": round(ms * 1e3 / steps, 3), "weight_copies": rot, "noise": noise,
            "traffic": recorded_traffic("gemv_m1_staged_kernel<1,0,4,0>")}


def run_prefill_repacked(q, steps, warmup, dist, peaks):
    """The prefill workload on Q4_0 weights repacked at load time."""
    import torch
    m, n, k = 512, 14336, 4096
    rot = copies_for(q4_weight_bytes(n, k) + m * k)
    wts, x = _quantized_weights(q, 11, n, k, m, rot, outlier_p=0.01)
    reps = [(q.repack_q4_0_gemm(wq), wd) for wq, wd in wts]
    del wts
    aq, ad = q.quantize_act_q8_0(_up(x))
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    ws = torch.empty((q.workspace_bytes(q.OP_GEMM, m, n, k),), dtype=torch.uint8, device="cuda")

    def step(i):
        wr, wd = reps[i % rot]
        q.gemm_q4_0_q8_0_repacked(wr, wd, aq, ad, y=y, workspace=ws)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    tops = dist.world * 2.0 * m * n * k * steps / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": "Q4_0xQ8_0 prefill GEMM m=512 K=4096 N=14336, 1% outliers x20 "
                        "(seed 11; weights repacked at load time)",
            "value": round(tops, 1), "unit": "TOPS (int ops, 2*m*n*k)",
            "frac_tensor": round(tops / dist.world / peak, 4), "peak": peak,
            **int8_fraction(tops / dist.world, peaks),
            "us_per_launch": round(ms * 1e3 / steps, 3), "weight_copies": rot, "noise": noise,
            "traffic": recorded_traffic("gemm_blocks_kernel<128,0,32,1>")}


def q8_weight_bytes(n, k):
    return n * k + 2 * n * (k // QK)


def _q8_weights(q, seed, n, k, m, copies, **kw):
    """As _quantized_weights, with Q8_0 weights (the activation recipe)."""
    from quantized_matmul_gb300 import synthetic
    w, x = synthetic.q4_0_case(seed, n, k, m, **kw)
    wdev = _up(w)
    w8, wd = q.quantize_weight_q8_0(wdev)
    del wdev
    return [(w8, wd)] + [(w8.clone(), wd.clone()) for _ in range(copies - 1)], x


def run_q8_gemv(q, steps, warmup, dist, peaks):
    """Q8_0 weights x Q8_0 decode GEMV at the 4096 x 4096 shape (seed 0)."""
    import torch
    n, k = 4096, 4096
    rot = copies_for(q8_weight_bytes(n, k))
    wts, x = _q8_weights(q, 0, n, k, 1, rot)
    aq, ad = q.quantize_act_q8_0(_up(x))
    y = torch.empty((1, n), dtype=torch.float32, device="cuda")

    def step(i):
        w8, wd = wts[i % rot]
        q.gemv_q8_0_q8_0(w8, wd, aq, ad, y=y, split_k=1)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    nbytes = q8_weight_bytes(n, k) + k + 2 * (k // QK) + 4 * n
    gbs = dist.world * nbytes * steps / (ms * 1e-3) / 1e9
    return {"workload": "Q8_0xQ8_0 GEMV m=1 K=4096 N=4096 (seed 0; Q8_0 weights)",
            "value": round(gbs, 1), "unit": "GB/s",
            "frac_hbm": round(gbs / dist.world / peaks["hbm_gbs"], 4),
            "us_per_launch": round(ms * 1e3 / steps, 3), "weight_copies": rot, "noise": noise,
            "traffic": recorded_traffic("gemv_q8_0_q8_0_kernel<1,2,0>"),
            "algorithmic_bytes_per_launch": nbytes}


def run_q8_prefill(q, steps, warmup, dist, peaks):
    """Q8_0 weights x Q8_0 prefill GEMM at the 512 x 14336 x 4096 shape."""
    import torch
    m, n, k = 512, 14336, 4096
    rot = copies_for(q8_weight_bytes(n, k) + m * k)
    wts, x = _q8_weights(q, 11, n, k, m, rot, outlier_p=0.01)
    aq, ad = q.quantize_act_q8_0(_up(x))
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    ws = torch.empty((q.workspace_bytes(q.OP_GEMM_Q8, m, n, k),), dtype=torch.uint8, device="cuda")

    def step(i):
        w8, wd = wts[i % rot]
        q.gemm_q8_0_q8_0(w8, wd, aq, ad, y=y, workspace=ws)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    tops = dist.world * 2.0 * m * n * k * steps / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": "Q8_0xQ8_0 prefill GEMM m=512 K=4096 N=14336, 1% outliers x20 "
                        "(seed 11; Q8_0 weights)",
            "value": round(tops, 1), "unit": "TOPS (int ops, 2*m*n*k)",
            "frac_tensor": round(tops / dist.world / peak, 4), "peak": peak,
            **int8_fraction(tops / dist.world, peaks),
            "us_per_launch": round(ms * 1e3 / steps, 3), "weight_copies": rot, "noise": noise,
            "traffic": recorded_traffic("gemm_blocks_kernel<128,0,64,0>")}


def run_q8_vocab(q, steps, warmup, dist, peaks, ms_list=(8, 16)):
    """Q8_0 weights x Q8_0 at the vocabulary shape (K=4096, N=128256, seed
    13) for a few tokens: the GEMM call, which takes the few-token product."""
    import torch
    n, k = 128256, 4096
    wts, x = _q8_weights(q, 13, n, k, max(ms_list), 1)
    w8, wd = wts[0]
    out = {"workload": "Q8_0xQ8_0 vocabulary projection K=4096 N=128256 (seed 13; Q8_0 "
                       "weights, 558.4 MB > 2x L2)", "m": {}}
    for m in ms_list:
        aq, ad = q.quantize_act_q8_0(_up(x[:m]))
        y = torch.empty((m, n), dtype=torch.float32, device="cuda")
        ws = torch.empty((q.workspace_bytes(q.OP_GEMM_Q8, m, n, k),), dtype=torch.uint8,
                         device="cuda")
        ms, noise = GraphTimer(lambda i: q.gemm_q8_0_q8_0(w8, wd, aq, ad, y=y, workspace=ws),
                               1).median(steps, warmup, dist)
        t = ms * 1e-3 / steps
        nbytes = q8_weight_bytes(n, k) + m * k + 2 * m * (k // QK) + 4 * m * n
        gb = dist.world * nbytes / t / 1e9
        out["m"][str(m)] = {"us": round(t * 1e6, 2), "GB/s": round(gb, 1), "noise": noise,
                            "frac_hbm": round(gb / dist.world / peaks["hbm_gbs"], 4),
                            "TOPS": round(dist.world * 2.0 * m * n * k / t / 1e12, 2),
                            "algorithmic_bytes_per_launch": nbytes}
        if m == 16:
            out["m"][str(m)]["traffic"] = recorded_traffic("gemm_small_m_kernel<32,1,2,0>")
    return out


def run_bitnet_batch(q, steps, warmup, dist, peaks, ms_list=(4, 8, 16, 32)):
    """BitNet 2560 -> 6912 (seed 3) for a few tokens on pre-quantized
    activations: qmm_bitnet_gemm (the warp-level few-token product for
    m <= 32) beside qmm_bitnet_gemv (m <= 16)."""
    import torch
    from quantized_matmul_gb300 import synthetic
    n, k = 6912, 2560
    t, x, absmean = synthetic.bitnet_case(3, n, k, max(ms_list))
    rot = copies_for(n * k // 4)
    tw = q.pack_ternary(_up(t))
    tws = [tw] + [tw.clone() for _ in range(rot - 1)]
    out = {"workload": "BitNet K=2560 N=6912 (seed 3), a few tokens, pre-quantized activations",
           "weight_copies": rot, "m": {}}
    for m in ms_list:
        aq, sc, sm = q.quantize_act_bitnet(_up(x[:m]))
        y = torch.empty((m, n), dtype=torch.float32, device="cuda")
        ws = torch.empty((q.workspace_bytes(q.OP_BITNET_GEMM, m, n, k),), dtype=torch.uint8,
                         device="cuda")
        paths = [("gemm", lambda i: q.bitnet_gemm(tws[i % rot], absmean, aq, sc, y=y,
                                                   workspace=ws))]
        if m <= 16:
            paths.append(("gemv", lambda i: q.bitnet_gemv(tws[i % rot], absmean, aq, sc, sm, y=y)))
        res = {}
        for name, fn in paths:
            ms, noise = GraphTimer(fn, rot).median(steps, warmup, dist)
            us = ms * 1e3 / steps
            res[name] = {"us": round(us, 2), "TOPS": round(dist.world * 2.0 * m * n * k / us / 1e6, 2),
                         "noise": noise}
        out["m"][str(m)] = res
    return out


def run_bitnet(q, steps, warmup, dist, peaks):
    """The BitNet decode step: per-row activation quantization + ternary
    GEMV in one call (qmm_linear_bitnet with programmatic dependent launch;
    at m = 1 a single kernel), from the f32 activation row to the f32
    output.  The GEMV alone on pre-quantized activations is reported beside
    it."""
    import torch
    from quantized_matmul_gb300 import synthetic
    n, k = 6912, 2560
    t, x, absmean = synthetic.bitnet_case(3, n, k, 1)
    rot = copies_for(n * k // 4)
    tw = q.pack_ternary(_up(t))
    tws = [tw] + [tw.clone() for _ in range(rot - 1)]
    xd = _up(x)
    aq = torch.empty((1, k), dtype=torch.int8, device="cuda")
    s = torch.empty((1,), dtype=torch.float32, device="cuda")
    asum = torch.empty((1,), dtype=torch.int32, device="cuda")
    y = torch.empty((1, n), dtype=torch.float32, device="cuda")

    def step(i):
        q.linear_bitnet(xd, tws[i % rot], absmean, y=y, pdl=True, aq=aq, act_scale=s, act_sum=asum)

    def gemv(i):
        q.bitnet_gemv(tws[i % rot], absmean, aq, s, asum, y=y)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    ms_g, _ = GraphTimer(gemv, rot).median(steps, warmup, dist)
    step_bytes = bitnet_step_bytes(1, n, k)
    gbs = dist.world * step_bytes * steps / (ms * 1e-3) / 1e9
    gbs_g = dist.world * bitnet_bytes(1, n, k) * steps / (ms_g * 1e-3) / 1e9
    return {"workload": "BitNet decode step m=1 K=2560 N=6912 (seed 3): per-row activation "
                        "quantization + ternary GEMV in one call (qmm_linear_bitnet, PDL; one "
                        "kernel at m=1, every CTA quantizing the row itself)",
            "value": round(gbs, 1), "unit": "GB/s",
            "frac_hbm": round(gbs / dist.world / peaks["hbm_gbs"], 4),
            "frac_hbm_nominal": round(gbs / dist.world / NOMINAL_HBM_GBS, 4),
            "us_per_step": round(ms * 1e3 / steps, 3), "algorithmic_bytes_per_step": step_bytes,
            "noise": noise,
            "gpu_launches_per_step": 1, "weight_copies": rot,
            "traffic": recorded_traffic("bitnet_linear_m1_kernel<3,8,1>"),
            "traffic_note": "DRAM bytes of one launch from the recorded ncu capture "
                            "(profiles/traffic.txt)",
            "gemv_alone": {"value": round(gbs_g, 1), "unit": "GB/s",
                           "frac_hbm": round(gbs_g / dist.world / peaks["hbm_gbs"], 4),
                           "us_per_launch": round(ms_g * 1e3 / steps, 3),
                           "algorithmic_bytes_per_launch": bitnet_bytes(1, n, k),
                           "traffic": recorded_traffic("bitnet_gemv_m1_kernel<1,8,0,0>")}}


def run_bitnet_prefill(q, steps, warmup, dist, peaks):
    import torch
    from quantized_matmul_gb300 import synthetic
    m, n, k = 2048, 6912, 2560
    t, x, absmean = synthetic.bitnet_case(3, n, k, m)
    tw = q.pack_ternary(_up(t))
    rot = copies_for(n * k // 4 + m * k)
    tws = [tw] + [tw.clone() for _ in range(rot - 1)]
    aq, s, _ = q.quantize_act_bitnet(_up(x))
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    ws = torch.empty((q.workspace_bytes(q.OP_BITNET_GEMM, m, n, k),), dtype=torch.uint8,
                     device="cuda")

    def step(i):
        q.bitnet_gemm(tws[i % rot], absmean, aq, s, y=y, workspace=ws)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    tops = dist.world * 2.0 * m * n * k * steps / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": "BitNet ternary prefill m=2048 K=2560 N=6912 (seed 3), tensor cores",
            "value": round(tops, 1), "unit": "TOPS (int ops, 2*m*n*k)",
            "frac_tensor": round(tops / dist.world / peak, 4), "peak": peak,
            "peak_note": "dense fp16/bf16 tensor peak (measured bf16 burst): codes - 1 and "
                         "int8 activations run exactly on tcgen05 kind::f16",
            "us_per_launch": round(ms * 1e3 / steps, 3), "weight_copies": rot, "noise": noise,
            "traffic": recorded_traffic("bitnet_gemm_kernel"),
            "traffic_note": "DRAM bytes of one launch from the recorded ncu capture "
                            "(profiles/traffic.txt); algorithmic: 4.4 MB codes + 10.5 MB fp16 "
                            "activations + 56.6 MB y (most of y is written back from L2 after "
                            "the kernel)"}


def run_prefill(q, steps, warmup, dist, peaks):
    import torch
    m, n, k = 512, 14336, 4096
    rot = copies_for(q4_weight_bytes(n, k) + m * k)
    wts, x = _quantized_weights(q, 11, n, k, m, rot, outlier_p=0.01)
    aq, ad = q.quantize_act_q8_0(_up(x))
    acts = [(aq, ad)] + [(aq.clone(), ad.clone()) for _ in range(rot - 1)]
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    ws = torch.empty((q.workspace_bytes(q.OP_GEMM, m, n, k),), dtype=torch.uint8, device="cuda")

    def step(i):
        wq, wd = wts[i % rot]
        a, d = acts[i % rot]
        q.gemm_q4_0_q8_0(wq, wd, a, d, y=y, workspace=ws)

    ms, noise = GraphTimer(step, rot).median(steps, warmup, dist)
    tops = dist.world * 2.0 * m * n * k * steps / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": "Q4_0xQ8_0 prefill GEMM m=512 K=4096 N=14336, 1% outliers x20 (seed 11)",
            "value": round(tops, 1), "unit": "TOPS (int ops, 2*m*n*k)",
            "frac_tensor": round(tops / dist.world / peak, 4), "peak": peak,
            "peak_note": "dense fp16/bf16 tensor peak (measured bf16 burst): the block sums run "
                         "on tcgen05 kind::f16 because sm_103a has no tcgen05 int8 MMA",
            **int8_fraction(tops / dist.world, peaks),
            "us_per_launch": round(ms * 1e3 / steps, 3), "weight_copies": rot, "noise": noise,
            "traffic": recorded_traffic("gemm_blocks_kernel<128,0,32,0>"),
            "traffic_note": "DRAM bytes of one launch from the recorded ncu capture "
                            "(profiles/traffic.txt); algorithmic: 33.0 MB weights + 2.1 MB "
                            "activations + 29.4 MB y (y is written back from L2 after the "
                            "kernel)"}


def int8_fraction(tops_per_gpu: float, peaks) -> dict:
    """The product's rate against the GPU's int8 tensor peak: the measured
    rate of mma.sync m16n8k32 s8, the only int8 tensor-core instruction
    sm_103a accepts (qmm_debug_mma_probe, timed in this run)."""
    p = peaks.get("int8_mma_tops")
    if not p:
        return {}
    return {"frac_int8": round(tops_per_gpu / p, 4), "int8_peak": round(p, 1),
            "int8_peak_note": "measured in this run: mma.sync m16n8k32 s8 x s8 -> s32 on every "
                              "SM (tcgen05.mma kind::i8 does not assemble for sm_103a)"}


def run_vocab(q, steps, warmup, dist, peaks, ms_list=(1, 8, 16, 32, 64, 128)):
    import torch
    n, k = 128256, 4096
    wts, x = _quantized_weights(q, 13, n, k, 128, 1)
    wq, wd = wts[0]
    out = {"workload": "Q4_0xQ8_0 vocabulary projection K=4096 N=128256 (seed 13), "
                       "weights 295.5 MB > 2x L2", "m": {},
           "paths": "gemv: qmm_gemv_q4_0_q8_0 with split_k=1 (the dp4a GEMV kernels); gemm: "
                    "qmm_gemm_q4_0_q8_0 (the few-token product for m <= 64, else tcgen05). "
                    "qmm_gemv_q4_0_q8_0 with split_k=0 takes the few-token product from m = 3 on"}
    for m in ms_list:
        aq, ad = q.quantize_act_q8_0(_up(x[:m]))
        y = torch.empty((m, n), dtype=torch.float32, device="cuda")
        ws = torch.empty((q.workspace_bytes(q.OP_GEMM, m, n, k),), dtype=torch.uint8,
                         device="cuda")
        res = {}
        paths = [("gemm", lambda i: q.gemm_q4_0_q8_0(wq, wd, aq, ad, y=y, workspace=ws))]
        if m <= 16:
            paths.insert(0, ("gemv", lambda i: q.gemv_q4_0_q8_0(wq, wd, aq, ad, y=y, split_k=1)))
        for name, fn in paths:
            ms, noise = GraphTimer(fn, 1).median(steps, warmup, dist)
            t = ms * 1e-3 / steps
            gb = dist.world * gemv_bytes(m, n, k) / t / 1e9
            res[name] = {"us": round(t * 1e6, 2), "GB/s": round(gb, 1), "noise": noise,
                         "frac_hbm": round(gb / dist.world / peaks["hbm_gbs"], 4),
                         "TOPS": round(dist.world * 2.0 * m * n * k / t / 1e12, 2)}
        if m == 16:
            res["gemm"]["traffic"] = recorded_traffic("gemm_small_m_kernel<16,1,2,0>")
        res["faster"] = min((r for r in res if r in ("gemv", "gemm")), key=lambda r: res[r]["us"])
        out["m"][str(m)] = res
    return out


# ---------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)

def _oracle_layer_set(row_fraction: float):
    import oracle
    from quantized_matmul_gb300 import synthetic
    mats = []
    for j, (n, k) in enumerate(LAYER_SET):
        w, x = synthetic.q4_0_case(j + 1, n, k, 1)
        rows = max(1, int(round(n * row_fraction)))
        wq, wd = oracle.quantize_q4_0(w[:rows])
        mats.append((n, k, rows, wq, wd, x))
    return mats


def _oracle_step(mats):
    import oracle
    moved = 0
    for n, k, rows, wq, wd, x in mats:
        aq, ad = oracle.quantize_q8_0(x)
        oracle.gemm_q4_0_q8_0(wq, wd, aq, ad)
        moved += linear_bytes(1, rows, k)  # the GPU arm's accounting, on the sampled rows
    return moved


def host_cores() -> list[int]:
    try:
        return sorted(os.sched_getaffinity(0))
    except AttributeError:
        return list(range(os.cpu_count() or 1))


def _oracle_step_threads(mats, threads: int, ex=None):
    """One layer-set step of the oracle with each matrix's rows split over
    `threads` threads of the executor `ex` (the oracle's C calls release the
    GIL): rows are independent, so the outputs are bit for bit those of one
    thread."""
    import oracle
    if threads <= 1 or ex is None:
        return _oracle_step(mats)
    moved = 0
    for n, k, rows, wq, wd, x in mats:
        aq, ad = oracle.quantize_q8_0(x)
        cuts = [rows * t // threads for t in range(threads + 1)]
        parts = [ex.submit(oracle.gemm_q4_0_q8_0, wq[a:b], wd[a:b], aq, ad)
                 for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
        for f in parts:
            f.result()
        moved += linear_bytes(1, rows, k)
    return moved


def _oracle_rate(mats, threads: int, budget_s: float, pin_core: int | None = None):
    """GB/s of repeated oracle steps for about budget_s seconds."""
    from concurrent.futures import ThreadPoolExecutor
    old = None
    if pin_core is not None:
        try:
            old = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {pin_core})
        except (AttributeError, OSError):
            old = None
    ex = ThreadPoolExecutor(threads) if threads > 1 else None
    try:
        _oracle_step_threads(mats, threads, ex)  # threads started, caches warm
        steps, moved, t0 = 0, 0, time.perf_counter()
        while True:
            moved += _oracle_step_threads(mats, threads, ex)
            steps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    finally:
        if ex is not None:
            ex.shutdown()
        if old is not None:
            os.sched_setaffinity(0, old)
    return moved / el / 1e9, steps, el


def guarded(fn):
    """A secondary measurement whose failure must not cost the contract line:
    its exception is recorded in its place.  (The same code fails the same
    way on every rank, so no rank waits in a collective the others skip.)"""
    try:
        return fn()
    except Exception as e:  # noqa: BLE001 - recorded, not hidden
        return {"error": f"{type(e).__name__}: {e}"[:400]}


# ---------------------------------------------------------------------------
# Result checksums and run identity

FNV64_OFFSET = 0xCBF29CE484222325  # FNV-1a, 64-bit (Fowler, Noll, Vo)
FNV64_PRIME = 0x100000001B3


def fnv1a64(data: bytes) -> str:
    h = FNV64_OFFSET
    for byte in data:
        h = ((h ^ byte) * FNV64_PRIME) & 0xFFFFFFFFFFFFFFFF
    return f"0x{h:016x}"


CHECK_ROWS, CHECK_N, CHECK_K = 512, 4096, 4096  # rows 0..511 of the 4096 x 4096 GEMV (seed 0)


def _check_inputs():
    from quantized_matmul_gb300 import synthetic
    w, x = synthetic.q4_0_case(0, CHECK_N, CHECK_K, 1)
    return np.ascontiguousarray(w[:CHECK_ROWS]), x


def gpu_checksums(q):
    """FNV-1a of integer results of the CUDA path on a fixed case: the Q8_0
    codes of the 4096-element activation row (seed 0) and the GEMV's int32
    block sums [1, 512, 128] against the first 512 rows of the 4096 x 4096
    weights, both quantized on the GPU.  Integer results are exact, so any
    machine (and the oracle) must give the same bytes."""
    import torch
    w, x = _check_inputs()
    wq, _ = q.quantize_weight_q4_0(_up(w))
    aq, _ = q.quantize_act_q8_0(_up(x))
    sumi = q.debug_block_sums(0, wq, aq)
    torch.cuda.synchronize()
    return {"q8_0_codes": fnv1a64(aq.cpu().numpy().tobytes()),
            "block_sums": fnv1a64(sumi.cpu().numpy().tobytes())}


def oracle_checksums():
    """The same two checksums from the oracle (CPU), quantizing the same f32
    inputs itself."""
    import oracle
    w, x = _check_inputs()
    wq, _ = oracle.quantize_q4_0(w)
    aq, _ = oracle.quantize_q8_0(x)
    return {"q8_0_codes": fnv1a64(np.ascontiguousarray(aq).tobytes()),
            "block_sums": fnv1a64(np.ascontiguousarray(oracle.block_sums(wq, aq)).tobytes())}


def run_identity():
    """The source the run was built from: the git commit where the checkout
    has one, else a SHA-256 over the native and Python sources."""
    import hashlib
    import subprocess
    try:
        sha = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                             text=True, timeout=10).stdout.strip()
    except (OSError, subprocess.SubprocessError):
        sha = ""
    h = hashlib.sha256()
    for sub in ("quantized_matmul_gb300/csrc", "quantized_matmul_gb300", "include", "oracle"):
        d = os.path.join(ROOT, sub)
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h", ".c", ".py")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + b"\0" + f.read())
    out = {"source_sha256": h.hexdigest()}
    if len(sha) == 40:
        out["git_commit"] = sha
    return out


def gpu_identity():
    import torch
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    return {"name": p.name, "compute_capability": f"{p.major}.{p.minor}",
            "sms": p.multi_processor_count, "memory_gib": round(p.total_memory / 2**30, 1)}


def cpu_baseline(budget_s: float, frac: float = 0.25):
    """The oracle as it stands on the host cores: one core (pinned) and all
    host cores (rows split over threads), each the median of three runs of
    about budget_s / 6 seconds over the same row sample."""
    mats = _oracle_layer_set(frac)
    cores = host_cores()
    each = max(budget_s / 6.0, 0.5)
    one = [_oracle_rate(mats, 1, each, pin_core=cores[0]) for _ in range(3)]
    allc = [_oracle_rate(mats, len(cores), each) for _ in range(3)]
    med1 = statistics.median(r[0] for r in one)
    medn = statistics.median(r[0] for r in allc)
    sample = (f"layer-set steps, each the Q8_0 quantization of all 7 activation rows plus the "
              f"scalar GEMV over the first {frac:.0%} of rows of every matrix; median of 3 runs "
              f"of ~{each:.1f} s each")
    return {"value": round(medn, 4), "unit": "GB/s", "cores": len(cores), "kind": "oracle",
            "host_cores": len(cores), "checksums": oracle_checksums(),
            "sample": sample + f", rows split over {len(cores)} threads",
            "runs": [round(r[0], 4) for r in allc],
            "one_core": {"value": round(med1, 4), "unit": "GB/s", "cores": 1,
                         "runs": [round(r[0], 4) for r in one],
                         "sample": sample + ", one thread pinned to one core"}}


def run_reference(args, dist):
    if dist.rank != 0:
        return
    # a 1% row sample calibrates the cost of a full step; each timed step then
    # takes a row sample sized so warm-up + steps finish within the budget
    from concurrent.futures import ThreadPoolExecutor
    cores = len(host_cores())
    ex = ThreadPoolExecutor(cores) if cores > 1 else None
    probe_frac = 0.01
    probe = _oracle_layer_set(probe_frac)
    _oracle_step_threads(probe, cores, ex)
    t0 = time.perf_counter()
    _oracle_step_threads(probe, cores, ex)
    full_s = (time.perf_counter() - t0) / probe_frac
    del probe
    frac = min(1.0, args.ref_budget / max(1, args.steps + args.warmup) / max(full_s, 1e-6))
    frac = max(frac, 1e-4)
    mats = _oracle_layer_set(frac)
    for _ in range(args.warmup):
        _oracle_step_threads(mats, cores, ex)
    t0 = time.perf_counter()
    moved = sum(_oracle_step_threads(mats, cores, ex) for _ in range(args.steps))
    el = time.perf_counter() - t0
    if ex is not None:
        ex.shutdown()
    value = moved / el / 1e9
    sample = (f"each step: Q8_0 quantization of all 7 activation rows + scalar GEMV over the "
              f"first {frac:.4%} of rows of every matrix of the layer set, rows split over "
              f"{cores} threads (all host cores)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / max(1, args.steps), 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": WORKLOAD_C2, "m": 1, "row_fraction": frac},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["qmm", "reference"], default="qmm")
    ap.add_argument("--configs", choices=["all", "main"], default="all",
                    help="'main' measures only the layer-set headline")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of oracle work for --impl reference (warm-up + steps)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for the cpu_baseline leg (0: skip it)")
    ap.add_argument("--only", choices=["gemv", "bitnet", "prefill", "vocab", "bitnet_prefill",
                                       "q8_gemv", "q8_prefill", "q8_vocab", "prefill_repacked",
                                       "bitnet_batch"],
                    default=None,
                    help="profiling aid: run only this workload (steps as given) and print "
                         "its result; the headline contract line is not produced")
    ap.add_argument("--vocab-m", default="1,8,16,32,64,128",
                    help="token counts of the vocabulary sweep (comma-separated, each <= 128)")
    ap.add_argument("--q8-vocab-m", default="8,16",
                    help="token counts of the Q8_0-weight vocabulary sweep (each <= 32)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    vocab_m = tuple(int(v) for v in args.vocab_m.split(","))
    q8_vocab_m = tuple(int(v) for v in args.q8_vocab_m.split(","))
    if not q8_vocab_m or any(not 1 <= v <= 32 for v in q8_vocab_m):
        ap.error("--q8-vocab-m takes token counts from 1 to 32")
    if not vocab_m or any(not 1 <= v <= 128 for v in vocab_m):
        ap.error("--vocab-m takes token counts from 1 to 128")
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
            return
        import torch
        torch.cuda.set_device(dist.local_rank)
        import quantized_matmul_gb300 as q
        q.load()  # the CUDA library; raises if it is missing
        peaks = load_peaks()
        # the int8 tensor peak the prefill products are reported against
        # (and the warp-level f16 rate beside it), measured now on this GPU
        peaks["int8_mma_tops"] = q.mma_probe_tops(0)
        peaks["f16_mma_sync_tflops"] = q.mma_probe_tops(1)
        if args.only:
            run = {"gemv": lambda: run_single_gemv(q, args.steps, args.warmup, dist, peaks),
                   "bitnet": lambda: run_bitnet(q, args.steps, args.warmup, dist, peaks),
                   "prefill": lambda: run_prefill(q, args.steps, args.warmup, dist, peaks),
                   "vocab": lambda: run_vocab(q, args.steps, args.warmup, dist, peaks, vocab_m),
                   "bitnet_prefill": lambda: run_bitnet_prefill(q, args.steps, args.warmup, dist,
                                                                peaks),
                   "q8_gemv": lambda: run_q8_gemv(q, args.steps, args.warmup, dist, peaks),
                   "q8_prefill": lambda: run_q8_prefill(q, args.steps, args.warmup, dist, peaks),
                   "q8_vocab": lambda: run_q8_vocab(q, args.steps, args.warmup, dist, peaks,
                                                    q8_vocab_m),
                   "bitnet_batch": lambda: run_bitnet_batch(q, args.steps, args.warmup, dist, peaks),
                   "prefill_repacked": lambda: run_prefill_repacked(q, args.steps, args.warmup,
                                                                    dist, peaks)}
            res = run[args.only]()
            if dist.rank == 0:
                print(json.dumps({"only": args.only, "result": res}), flush=True)
            return
        main_res = run_layer_set(q, args, dist, peaks)
        configs = {"layer_set_variants": main_res["variants"]}
        if args.configs == "all":
            short = max(200, min(args.steps, 4000))
            long_ = max(50, short // 20)
            table = [
                ("gemv_4096x4096", lambda: run_single_gemv(q, short * 5, args.warmup, dist, peaks)),
                ("bitnet_2560x6912", lambda: run_bitnet(q, short * 5, args.warmup, dist, peaks)),
                ("prefill_512x14336x4096", lambda: run_prefill(q, long_, 10, dist, peaks)),
                ("bitnet_prefill_2048x6912x2560",
                 lambda: run_bitnet_prefill(q, long_, 10, dist, peaks)),
                ("bitnet_batch_2560x6912",
                 lambda: run_bitnet_batch(q, max(200, short // 4), 10, dist, peaks)),
                ("vocab_4096x128256", lambda: run_vocab(q, long_, 10, dist, peaks, vocab_m)),
                ("prefill_repacked_512x14336x4096",
                 lambda: run_prefill_repacked(q, long_, 10, dist, peaks)),
                ("q8_0_gemv_4096x4096", lambda: run_q8_gemv(q, short * 5, args.warmup, dist, peaks)),
                ("q8_0_prefill_512x14336x4096", lambda: run_q8_prefill(q, long_, 10, dist, peaks)),
                ("q8_0_vocab_4096x128256",
                 lambda: run_q8_vocab(q, long_, 10, dist, peaks, q8_vocab_m)),
            ]
            for name, fn in table:
                configs[name] = guarded(fn)
        cpu = cpu_baseline(args.cpu_budget) if dist.rank == 0 and args.cpu_budget > 0 else None
        checks = None
        if dist.rank == 0:
            gpu_sums = guarded(lambda: gpu_checksums(q))
            checks = {"case": f"Q4_0 GEMV {CHECK_N}x{CHECK_K} (seed 0), weight rows 0..{CHECK_ROWS - 1}, "
                              f"m = 1: FNV-1a-64 of the Q8_0 codes and of the int32 block sums",
                      "gpu": gpu_sums}
            if cpu is not None:  # the oracle's own checksums come with its baseline
                checks["oracle"] = cpu.pop("checksums")
                checks["match"] = checks["oracle"] == gpu_sums
        if dist.rank == 0:
            line = {
                "metric": METRIC, "value": round(main_res["value"], 1), "unit": "GB/s",
                "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(main_res["ms"], 6), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int8",
                "data": "synthetic (seeded SplitMix64 + Box-Muller, weights quantized on the GPU)",
                "config": {"workload": WORKLOAD_C2, "m": 1,
                           "parallelism": f"replicas x{dist.world}",
                           "weight_bytes_per_step": main_res["set_bytes"],
                           "algorithmic_bytes_per_step": main_res["step_bytes"],
                           "l2": f"inputs larger than L2: rotating {main_res['rot']} copies of the "
                                 f"layer-set weights "
                                 f"({main_res['rot'] * main_res['set_bytes'] / 1e6:.0f} MB > "
                                 f"129 MB L2)",
                           "timing": "replays of CUDA graphs of 32 consecutive steps (plus one "
                                     "for the remainder), CUDA events on the launching stream"},
                "clocks": main_res["clocks"],
                "roofline": main_res["roofline"],
                "cpu_baseline": cpu,
                "e2e": main_res["e2e"],
                "gpu_launches": main_res["launches"],
                "noise": main_res["noise"],
                "frac_hbm_step": round(main_res["value"] / dist.world / peaks["hbm_gbs"], 4),
                "frac_hbm_step_nominal": round(main_res["value"] / dist.world / NOMINAL_HBM_GBS, 4),
                "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                          "source": peaks["source"], "nominal_hbm_gbs": NOMINAL_HBM_GBS,
                          "int8_mma_sync_tops": round(peaks["int8_mma_tops"], 1),
                          "f16_mma_sync_tflops": round(peaks["f16_mma_sync_tflops"], 1),
                          "mma_sync_note": "measured in this run with qmm_debug_mma_probe (warp-"
                                           "level MMA on every SM); int8 is the GPU's only int8 "
                                           "tensor path on sm_103a"},
                "configs": configs,
                "checks": checks,
                "gpu": gpu_identity(),
                "build": run_identity(),
            }
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
