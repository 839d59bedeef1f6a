"""Throughput of the tensor-parallel MLP block on GB300 (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole hot path over one batch: for the default
workload ``sp_block_fwd_bwd`` (T=8192 tokens in N=8 sequence chunks, d=4096,
F=16384) that is LayerNorm+gather, the column-parallel GEMM with bias+GeLU,
the row-parallel GEMM with the in-kernel shard reduction and fused
reduce-scatter store, then the backward on the forward's saved activations
(Xg, H, Hpre): dY B^T * GeLU', dB = H^T dY, dA = Xg^T dHpre, dXg = dHpre A^T
and the LayerNorm backward.
Every kernel is timed with CUDA events on the stream it is launched on; a GEMM
timed over less than a second is compared with the measured burst bf16 peak,
a longer one with the sustained peak, and also with the peak at the SM clock
the run held.  ``step_ms`` gives the p10 / median / p90 of the timed steps.
``e2e`` repeats the step through the block calls of the C ABI with the
activations copied from / to pinned host memory inside the timed region.
After the step, ``other_rows`` times the rest of the hot path on the same
shapes and the two forward-only workloads that carry the d = 4096 and d = 8192
forward GEMM rates (``mlp7b_fwd``, ``sp_large_fwd``).
The ``reference`` implementation is the CPU fp64 oracle on a bounded sample
of the same workload.
"""
import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tensor_transformer_mlp_tp_gb300 import inputs  # noqa: E402

METRIC = "TP-MLP block bf16 TFLOP/s and tokens/s at 1 GB300; % of dense BF16 / HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# A timed region shorter than this is compared with the burst peak (a cuBLAS GEMM timed alone), a longer
# one with the sustained peak (the same GEMM back to back for seconds, under the power cap).
SUSTAINED_AFTER_S = 1.0
# Dense bf16 tcgen05 rate per SM and clock: one 128 x 128 x 16 UMMA (524288 flops) per 64 cycles on an SM
# (a probe of the MMA alone on resident operands), i.e. 8192 flop/clk/SM.
BF16_FLOP_PER_CLK_SM = 8192.0


def tensor_peak(pk, region_s, dtype_factor=1.0):
    """(peak TFLOP/s, description) for a kernel timed over a region of `region_s` seconds: the measured burst
    peak below SUSTAINED_AFTER_S, the sustained one above; `dtype_factor` scales it (2 for FP8: the nominal
    dense FP8 : BF16 ratio)."""
    sustained = region_s >= SUSTAINED_AFTER_S and "bf16_tflops_sustained" in pk
    base = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    kind = "sustained" if sustained else "burst"
    if dtype_factor != 1.0:
        kind = f"{dtype_factor:g} x bf16 {kind}"
    return base * dtype_factor, kind


def clock_peak(sm_count, sm_mhz, dtype_factor=1.0):
    """Dense tensor peak (TFLOP/s) at the SM clock the run actually held: flop/clk/SM x SMs x clock."""
    if not sm_mhz or not sm_count:
        return None
    return BF16_FLOP_PER_CLK_SM * dtype_factor * sm_count * sm_mhz * 1e6 / 1e12


def percentiles(ms):
    """p10 / median / p90 of per-step times (ms)."""
    a = np.sort(np.asarray(ms, dtype=np.float64))
    return {"p10": round(float(np.percentile(a, 10)), 4), "median": round(float(np.median(a)), 4),
            "p90": round(float(np.percentile(a, 90)), 4)}


_GEMM_SOURCES = ("common.h", "ptx.cuh", "debug_bounds.cuh", "fp8.cuh", "philox.cuh", "launch.h", "gemm_tc.cuh",
                 "gemm_tc2.cuh", "gemm_tc.cu")
_ROW_SOURCES = ("common.h", "ptx.cuh", "debug_bounds.cuh", "fp8.cuh", "philox.cuh", "launch.h", "rowwise.cu")


def kernel_source_digest(segment=None):
    """Short sha256 of the CUDA sources a segment's kernels are built from (all sources without a segment);
    keys the committed ncu traffic table."""
    csrc = os.path.join(ROOT, "tensor_transformer_mlp_tp_gb300", "csrc")
    if segment is None:
        files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    else:
        files = _GEMM_SOURCES if segment.startswith("gemm") else _ROW_SOURCES
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(segment, workload=None):
    """DRAM bytes per launch of `segment` from the committed ncu capture, or None if its kernels changed since."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    entry = d.get("segments", {}).get(segment)
    if entry is None or entry.get("source_digest") != kernel_source_digest(segment):
        return None
    if workload is not None and d.get("workload") != workload:
        return None
    return entry.get("bytes_per_launch")


def max_over_ranks(value, dist):
    """The largest `value` over all ranks (every rank gets it); the value itself without a process group."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_step, steps, world, max_ms):
    """Work of all ranks (each rank does `work_per_step` per step) per second of the slowest rank."""
    return work_per_step * steps * world / (max_ms * 1e-3)


def useful_flops(w):
    """Algorithmic GEMM flops of one step: 2 T d F per GEMM; 2 forward GEMMs, 4 backward GEMMs."""
    per_gemm = 2.0 * w.T * w.d * w.F
    return per_gemm * (6 if w.backward else 2)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="tpmlp_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    @staticmethod
    def _epoch(stamp):
        import datetime
        try:
            return time.mktime(datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timetuple()) + \
                float("0." + stamp.rsplit(".", 1)[1])
        except (ValueError, IndexError):
            return None

    def _rows(self):
        if getattr(self, "_cache", None) is None:
            rows = []
            if self.proc is not None and os.path.exists(self.path):
                with open(self.path) as fh:
                    for line in fh:
                        parts = [x.strip() for x in line.split(",")]
                        if len(parts) >= 9:
                            rows.append(parts)
                os.unlink(self.path)
            self._cache = rows
        return self._cache

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in samples taken between t0 and t1 (epoch seconds)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self._rows()
        if t0 is not None:
            inside = [r for r in rows if (lambda e: e is not None and t0 - 0.1 <= e <= t1 + 0.1)(self._epoch(r[0]))]
            rows = inside or rows[-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- oracle (CPU) leg

_SAMPLE_CACHE = {}


def _cached_draw(w, name, seed, rows=None):
    key = (w.name, name, seed, None if rows is None else (int(rows[0]), len(rows)))
    if key not in _SAMPLE_CACHE:
        _SAMPLE_CACHE[key] = inputs.draw(w, name, seed, rows=rows)
    return _SAMPLE_CACHE[key]


def oracle_sample(w, seed=0, tokens=None):
    """Run the oracle on `tokens` rows of workload `w` (for the SP block: the first tokens/N rows of every
    chunk) with the full weights; returns (seconds of oracle work, tokens, flops)."""
    import oracle

    N = w.N
    tokens = tokens or w.T
    rows_per_chunk = max(1, tokens // N) if w.sp else tokens
    tok = rows_per_chunk * N if w.sp else tokens
    if w.sp:
        # the same chunk-local rows of every chunk
        sel = np.concatenate([np.arange(j * w.rows_per_chunk, j * w.rows_per_chunk + rows_per_chunk)
                              for j in range(N)])
    else:
        sel = np.arange(tok)
    X = _cached_draw(w, "X", seed, rows=sel)[1]
    A = _cached_draw(w, "A", seed)[1]
    B = _cached_draw(w, "B", seed)[1]
    b = _cached_draw(w, "bias", seed)
    b = None if b is None else b[1]
    if w.sp:
        g = _cached_draw(w, "gamma", seed)[1]
        be = _cached_draw(w, "beta", seed)[1]
        chunks = [X[j * rows_per_chunk:(j + 1) * rows_per_chunk] for j in range(N)]
        dyc = None
        if w.backward:
            dY = _cached_draw(w, "dY", seed, rows=sel)[1]
            dyc = [dY[j * rows_per_chunk:(j + 1) * rows_per_chunk] for j in range(N)]
        t0 = time.perf_counter()
        oracle.sp_forward(chunks, g, be, 1e-5, A, B, b, N)
        if w.backward:
            oracle.sp_backward(chunks, g, be, 1e-5, A, B, b, dyc, N)
    else:
        t0 = time.perf_counter()
        oracle.mlp_tp(X, A, B, b, N)
    dt = time.perf_counter() - t0
    flops = 2.0 * tok * w.d * w.F * (6 if w.backward else 2)
    return dt, tok, flops


def cpu_baseline_configs(tokens=64):
    """The oracle timed on a bounded sample of every configuration (the full tiny fp32 one; `tokens` rows of
    the others, with their full weights, drawn by the host generator), on the host cores: seconds, tokens,
    flops and TFLOP/s per configuration."""
    out = {}
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    for num, name in CONFIGS.items():
        w = inputs.WORKLOADS[name]
        t0 = time.perf_counter()
        dt, tok, fl = oracle_sample(w, tokens=w.T if w.dtype == "fp32" else tokens)
        out[name] = {"config": num, "oracle_s": round(dt, 3), "tokens": tok, "TFLOP/s": round(fl / dt / 1e12, 4),
                     "draw_s": round(time.perf_counter() - t0 - dt, 1), "cores": cores,
                     "work": "forward + backward" if w.backward else "forward"}
    return out


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    tokens = args.oracle_tokens
    for _ in range(args.warmup):
        oracle_sample(w, tokens=tokens)
    times, tok, flops = [], 0, 0.0
    for _ in range(args.steps):
        dt, tok, flops = oracle_sample(w, tokens=tokens)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"{tok} of {w.T} tokens ({tok // w.N if w.sp else tok} rows per chunk) with the full "
              f"d={w.d}, F={w.F} weights, numpy float64 (BLAS matmul on {cores} threads)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "tokens_per_s": tok * args.steps / total,
            "config": {"workload": w.name, "tokens": w.T, "d": w.d, "ffn": w.F, "n_shards": w.N,
                       "sample_tokens": tok},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU leg

class Step:
    """Device buffers of one workload and the sequence of ABI step calls of one step."""

    def __init__(self, w, torch, binding, seed=0, on_device=False):
        """Inputs from the seeded host generator of `inputs` (the parity tests' recipe), or with `on_device`
        from torch's seeded device generator with the same distributions (fast for the largest weights)."""
        self.w, self.torch, self.b = w, torch, binding
        dev = "cuda"
        T, d, F, N = w.T, w.d, w.F, w.N
        gen = None
        if on_device:
            gen = torch.Generator(device=dev)
            gen.manual_seed(seed)

        def up(name):
            if on_device:
                dist = w.dists.get(name)
                if dist is None:
                    return None
                shape = inputs.tensor_shape(w, name)
                if dist == "zero":
                    return torch.zeros(shape, dtype=torch.bfloat16, device=dev)
                t = torch.empty(shape, dtype=torch.float32, device=dev).normal_(dist[0], dist[1], generator=gen)
                return t.to(torch.bfloat16)  # round to nearest even, as the host recipe
            r = inputs.draw(w, name, seed)
            if r is None:
                return None
            return torch.from_numpy(np.ascontiguousarray(r[0]).view(np.int16)).view(torch.bfloat16).to(dev)

        self.X = up("X")
        self.A = up("A")
        self.B = up("B")
        self.bias = up("bias")
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.H = torch.empty(T, F, **bf)
        self.Y = torch.empty(T, d, **bf)
        self.rows = T // N
        if w.sp:
            self.gamma, self.beta = up("gamma"), up("beta")
            self.Xg = torch.empty(T, d, **bf)
            self.Xc = list(self.X.split(self.rows))
            self.Yc = list(self.Y.split(self.rows))
        if w.backward:
            self.dY = up("dY")
            self.dYc = list(self.dY.split(self.rows))
            self.Hpre = torch.empty(T, F, **bf)
            self.dHpre = torch.empty(T, F, **bf)
            self.dXg = torch.empty(T, d, **bf)
            self.dX = torch.empty(T, d, **bf)
            self.dXc = list(self.dX.split(self.rows))
            self.dA = torch.empty(d, F, **bf)
            self.dB = torch.empty(F, d, **bf)
            self.dgamma = torch.empty(d, dtype=torch.float32, device=dev)
            self.dbeta = torch.empty(d, dtype=torch.float32, device=dev)
            self.lnws = binding.workspace(binding.make_shape(T, d, F, N), binding.OP_LN_BWD)

    def kernels(self):
        """(name, launches, algorithmic work per launch, unit) of each timed segment of a step."""
        return Step.kernels_of(self.w)

    @staticmethod
    def kernels_of(w):
        g = 2.0 * w.T * w.d * w.F
        ln = 2.0 * w.T * w.d * 2          # read x, write y (bf16)
        segs = []
        if w.sp:
            segs.append(("layernorm_gather", 1, ln, "B"))
        segs += [("gemm1_bias_gelu", 1, g, "F"), ("gemm2_shard_accum" + ("_rs_store" if w.sp else ""), 1, g, "F")]
        if w.backward:
            segs += [("gemm_dh_geluprime", 1, g, "F"), ("gemm_wgrad_b", 1, g, "F"),
                     ("gemm_wgrad_a", 1, g, "F"), ("gemm_dx_shard_accum", 1, g, "F"),
                     ("layernorm_backward", 2, 3.0 * w.T * w.d * 2, "B")]
        return segs

    def run(self, ev=None):
        """Launch one step; if `ev` (a list of events) is given, record ev[i] after segment i (ev[0] before)."""
        b, w, N = self.b, self.w, self.w.N
        rec = (lambda i: ev[i].record()) if ev is not None else (lambda i: None)
        i = 0
        rec(i)
        if w.sp:
            b.tpmlp_layernorm_gather(self.Xc, self.gamma, self.beta, N, self.Xg)
            i += 1; rec(i)
            x_in = self.Xg
        else:
            x_in = self.X
        b.tpmlp_gemm1_bias_gelu(x_in, self.A, self.bias, N, self.H, self.Hpre if w.backward else None)
        i += 1; rec(i)
        if w.sp:
            b.tpmlp_gemm2_shard_accum(self.H, self.B, N, Y_chunks=self.Yc)
        else:
            b.tpmlp_gemm2_shard_accum(self.H, self.B, N, Y=self.Y)
        i += 1; rec(i)
        if w.backward:
            # the forward's gathered LayerNorm output Xg, H and Hpre are the saved activations
            b.tpmlp_gemm_dh_geluprime(self.dY, self.B, self.Hpre, N, self.dHpre)
            i += 1; rec(i)
            b.tpmlp_gemm_wgrad_b(self.H, self.dY, N, self.dB)
            i += 1; rec(i)
            b.tpmlp_gemm_wgrad_a(self.Xg, self.dHpre, N, self.dA)
            i += 1; rec(i)
            b.tpmlp_gemm_dx_shard_accum(self.dHpre, self.A, N, self.dXg)
            i += 1; rec(i)
            b.tpmlp_layernorm_backward(self.Xc, self.gamma, self.dXg, N, self.dXc, self.dgamma, self.dbeta,
                                       ws=self.lnws)
            i += 1; rec(i)
        return i

    def launches_per_step(self):
        return sum(n for _, n, _, _ in self.kernels())


def e2e_what(w):
    calls = ("tpmlp_sp_forward" if w.sp else "tpmlp_forward") + (" + tpmlp_sp_backward" if w.backward else "")
    io = ("X, dY", "Y, dX") if w.backward else ("X", "Y")
    return (f"block calls ({calls}) with {io[0]} copied from pinned host memory and {io[1]} copied back every step "
            "inside the timed region; inputs go up one step ahead on one copy stream and outputs come back on "
            "another, overlapping the kernels (X, dY and Y double-buffered on the device); weights"
            + (" and their gradients" if w.backward else "") + " stay in HBM")


def run_e2e(step, args, torch, binding):
    """The same step through the block calls, with each step's activations copied from pinned host memory and
    its outputs copied back inside the timed region.  Inputs go up on one copy stream into a double buffer, one
    step ahead (step k+1's X and dY while step k computes); outputs come back on a second copy stream (Y while
    the backward runs, dX while the next forward runs)."""
    w = step.w
    N = w.N
    X_h = step.X.cpu().pin_memory()
    Y_h = torch.empty_like(step.Y, device="cpu").pin_memory()
    h2d = X_h.numel() * 2
    d2h = Y_h.numel() * 2
    if w.backward:
        dY_h = step.dY.cpu().pin_memory()
        dX_h = torch.empty_like(step.dX, device="cpu").pin_memory()
        h2d += dY_h.numel() * 2
        d2h += dX_h.numel() * 2
    Xd = [torch.empty_like(step.X) for _ in range(2)]
    dYd = [torch.empty_like(step.dY) for _ in range(2)] if w.backward else None
    # Y double-buffered too: without a backward between them, a forward would otherwise wait for the
    # previous step's Y to reach the host
    Yd = [step.Y, torch.empty_like(step.Y)]
    Ycd = [list(y.split(step.rows)) for y in Yd] if w.sp else None
    shape = binding.make_shape(w.T, w.d, w.F, N)
    ws_f = binding.workspace(shape, binding.OP_SP_FWD if w.sp else binding.OP_FWD)
    ws_b = binding.workspace(shape, binding.OP_SP_BWD) if w.backward else None
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    used = [ev(), ev()]          # buffer b free again (its step's last kernel done)
    in_x, in_dy = [ev(), ev()], [ev(), ev()]  # buffer b holds its step's inputs
    y_out, dx_out = [ev(), ev()], ev()  # Y (buffer b) / dX copied to the host (may be overwritten)
    # a step's forward / backward done (re-recorded every step: a wait takes the event's latest record)
    fwd_done, bwd_done = ev(), ev()
    for e in used + in_x + in_dy + y_out + [dx_out]:
        e.record(comp)

    def inputs_up(k):
        b = k % 2
        up.wait_event(used[b])
        with torch.cuda.stream(up):
            Xd[b].copy_(X_h, non_blocking=True)
            in_x[b].record(up)
            if w.backward:
                dYd[b].copy_(dY_h, non_blocking=True)
                in_dy[b].record(up)

    def one(k, last):
        b = k % 2
        if not last:
            inputs_up(k + 1)
        comp.wait_event(in_x[b])
        comp.wait_event(y_out[b])
        if w.sp:
            binding.tpmlp_sp_forward(list(Xd[b].split(step.rows)), step.gamma, step.beta, step.A, step.B, N,
                                     Ycd[b], bias=step.bias, Hpre_out=step.Hpre if w.backward else None,
                                     H_out=step.H if w.backward else None, Xg_out=step.Xg if w.backward else None,
                                     ws=ws_f)
        else:
            binding.tpmlp_forward(Xd[b], step.A, step.B, step.bias, N, Yd[b], ws=ws_f)
        fwd_done.record(comp)
        down.wait_event(fwd_done)
        with torch.cuda.stream(down):
            Y_h.copy_(Yd[b], non_blocking=True)
            y_out[b].record(down)
        if w.backward:
            comp.wait_event(in_dy[b])
            comp.wait_event(dx_out)
            binding.tpmlp_sp_backward(list(Xd[b].split(step.rows)), step.gamma, step.beta, step.A, step.B,
                                      step.Hpre, list(dYd[b].split(step.rows)), N, step.dXc, step.dA, step.dB,
                                      step.dgamma, step.dbeta, bias=step.bias, H=step.H, Xg=step.Xg, ws=ws_b)
            bwd_done.record(comp)
            down.wait_event(bwd_done)
            with torch.cuda.stream(down):
                dX_h.copy_(step.dX, non_blocking=True)
                dx_out.record(down)
        used[b].record(comp)

    def run(n):
        inputs_up(0)
        for k in range(n):
            one(k, k == n - 1)

    run(max(1, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    up.wait_event(e0)
    run(args.steps)
    comp.wait_event(y_out[0])
    comp.wait_event(y_out[1])
    comp.wait_event(dx_out)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    return ms, h2d, d2h


def time_calls(torch, fn, reps, warmup=3):
    """Average ms of `fn` over `reps` back-to-back calls, CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# Pause before a row kernel is timed alone: after seconds of GEMMs the GPU sits at its power cap and its SM
# clock needs about 100 ms to recover, and the row kernels' time follows the SM clock.
SETTLE_S = 0.3


def time_graph(torch, fn, reps, warmup=3, settle=SETTLE_S):
    """Average ms of `fn` over `reps` back-to-back calls captured in one CUDA graph and replayed: the kernels'
    own time without the host's launch cost between them (a Python call through the C ABI takes about
    15 us of host time, more than half of a 25 us row kernel)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    time.sleep(settle)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del g
    return ms


def hbm_row(nb, ms_graph, ms_eager, pk, **extra):
    """A row kernel's rates: algorithmic bytes per launch over the graph-timed and the eager time."""
    gbs = lambda ms: nb / (ms * 1e-3) / 1e9
    out = {"ms": round(ms_graph, 4), "GB/s": round(gbs(ms_graph), 1), "frac": round(gbs(ms_graph) / pk["hbm_gbs"], 3),
           "timing": "CUDA graph of back-to-back launches", "eager_ms": round(ms_eager, 4),
           "eager_frac": round(gbs(ms_eager) / pk["hbm_gbs"], 3), "bytes_per_launch": nb}
    out.update(extra)
    return out


def run_fp8_step(step, torch, binding, pk):
    """The FP8 path on the step's shapes: the E4M3 forward (weight casts, E4M3 LayerNorm, both E4M3 GEMMs),
    the backward with E5M2 gradients (dY casts, weight casts, the E5M2 GeLU' GEMM, three byte transposes,
    three FP8 GEMMs, the bf16 LayerNorm backward) and both delayed-scale updates, timed as a whole and per
    GEMM.  The FP8 tensor peak is the measured burst bf16 peak (each GEMM is timed over ten calls) times the
    nominal dense FP8 : BF16 ratio of 2."""
    w = step.w
    T, d, F, N = w.T, w.d, w.F, w.N
    u8 = dict(dtype=torch.uint8, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    fwd = binding.fp8_state(torch.ones(4, device="cuda"), torch.zeros(4, device="cuda"),
                            torch.zeros(4, 16, device="cuda"))
    grad = binding.fp8_state(torch.ones(2, device="cuda"), torch.zeros(2, device="cuda"),
                             torch.zeros(2, 16, device="cuda"))
    shape = binding.make_shape(T, d, F, N)
    wsf = binding.workspace(shape, binding.OP_SP_FWD_FP8)
    wsb = binding.workspace(shape, binding.OP_SP_BWD_FP8)
    Hpre, Xq, Hq = torch.empty(T, F, **bf), torch.empty(T, d, **u8), torch.empty(T, F, **u8)
    dA, dB, db = torch.empty(d, F, **bf), torch.empty(F, d, **bf), torch.empty(F, **bf)
    dga, dbe = torch.empty(d, device="cuda"), torch.empty(d, device="cuda")

    def forward():
        binding.tpmlp_sp_forward_fp8(step.Xc, step.gamma, step.beta, step.A, step.B, N, step.Yc, fwd, bias=step.bias,
                                     Hpre_out=Hpre, Xq_out=Xq, Hq_out=Hq, ws=wsf)

    def train_step():
        forward()
        binding.tpmlp_sp_backward_fp8(step.Xc, step.gamma, step.A, step.B, Hpre, Xq, Hq, step.dYc, N, fwd, grad,
                                      step.dXc, dA, dB, dga, dbe, dbias=db, ws=wsb)
        binding.tpmlp_fp8_update_scales(fwd)

    def forward_only():
        forward()
        binding.tpmlp_fp8_update_scales(fwd)

    # calibrate: the first steps fill the amax histories, so the timed steps run on delayed scales of
    # the real amaxes
    for _ in range(16):
        train_step()
    ms_step = time_calls(torch, train_step, 10)
    ms_fwd = time_calls(torch, forward_only, 10)
    sc, am = fwd._tensors[0], fwd._tensors[1]
    gsc, gam = grad._tensors[0], grad._tensors[1]
    AqT, BqT = torch.empty(F, d, **u8), torch.empty(d, F, **u8)
    ms_ca = time_calls(torch, lambda: binding.tpmlp_cast_e4m3(step.A, sc[1:2], AqT, am[1:2], transpose=True), 10)
    ms_cb = time_calls(torch, lambda: binding.tpmlp_cast_e4m3(step.B, sc[2:3], BqT, am[2:3], transpose=True), 10)
    ms_g1 = time_calls(torch, lambda: binding.tpmlp_gemm1_e4m3(Xq, AqT, step.bias, N, sc[0:1], sc[1:2], sc[3:4], Hq,
                                                                am[3:4]), 10)
    ms_g2 = time_calls(torch, lambda: binding.tpmlp_gemm2_e4m3(Hq, BqT, N, sc[3:4], sc[2:3], Y_chunks=step.Yc), 10)
    dYq, Bq, dHq = torch.empty(T, d, **u8), torch.empty(F, d, **u8), torch.empty(T, F, **u8)
    binding.tpmlp_cast_e5m2(step.dY, gsc[0:1], dYq, gam[0:1])
    binding.tpmlp_cast_e4m3(step.B, sc[2:3], Bq, am[2:3])
    ms_dh = time_calls(torch, lambda: binding.tpmlp_gemm_dh_geluprime_e5m2(dYq, Bq, Hpre, N, gsc[0:1], sc[2:3],
                                                                            gsc[1:2], dHq, gam[1:2]), 10)
    HqT, dYqT = torch.empty(F, T, **u8), torch.empty(d, T, **u8)
    ms_tr = time_calls(torch, lambda: binding.tpmlp_transpose_bytes(Hq, HqT), 10)
    binding.tpmlp_cast_e5m2(step.dY, gsc[0:1], dYqT, gam[0:1], transpose=True)
    ms_wb = time_calls(torch, lambda: binding.tpmlp_gemm_fp8(HqT, binding.E4M3, dYqT, binding.E5M2, sc[3:4],
                                                              gsc[0:1], dB), 10)
    g = 2.0 * T * d * F
    # each GEMM is timed over ten calls (well under a second): the burst peak, doubled for FP8
    peak8, peak8_kind = tensor_peak(pk, 0.0, dtype_factor=2.0)
    tf = lambda ms: round(g / (ms * 1e-3) / 1e12, 1)
    kern = lambda ms: {"ms": round(ms, 4), "TFLOP/s": tf(ms), "frac": round(tf(ms) / peak8, 3)}
    return {"step_ms": round(ms_step, 4), "step_TFLOP/s": round(6 * g / (ms_step * 1e-3) / 1e12, 1),
            "forward_ms": round(ms_fwd, 4), "forward_TFLOP/s": round(2 * g / (ms_fwd * 1e-3) / 1e12, 1),
            "what": "tpmlp_sp_forward_fp8 + tpmlp_sp_backward_fp8 + tpmlp_fp8_update_scales (E4M3 forward, E5M2 "
                    "gradients, delayed scaling), the flops of the six GEMMs over the whole step",
            "gemm1_e4m3": kern(ms_g1), "gemm2_e4m3": kern(ms_g2), "dh_geluprime_e5m2": kern(ms_dh),
            "wgrad_b_e4m3_e5m2": kern(ms_wb),
            "cast_weights_transposed_ms": round(ms_ca + ms_cb, 4),
            "cast_weights_GB/s": round(3.0 * 2 * d * F / ((ms_ca + ms_cb) * 1e-3) / 1e9, 1),
            "transpose_H_ms": round(ms_tr, 4), "transpose_H_GB/s": round(2.0 * T * F / (ms_tr * 1e-3) / 1e9, 1),
            "peak_fp8_tflops": round(peak8, 1),
            "peak_kind": f"measured {peak8_kind} (the nominal dense FP8 : BF16 ratio is 2)"}


def run_attention(step, torch, binding, pk):
    """The tensor-parallel attention block on the step's width: d / 128 heads of 128 split over the N
    shards, the step's tokens as 2 sequences (sequence-major), causal; the attention core and the whole
    block (projection GEMM, core, output projection with the shard sum) timed on their own."""
    w = step.w
    d, N = w.d, w.N
    H, B = d // 128, 2
    S = w.T // B
    T = S * B
    bf = dict(dtype=torch.bfloat16, device="cuda")
    X = step.X[:T]
    Wqkv = torch.empty(d, 3 * d, **bf).normal_(0.0, d ** -0.5)
    Wo = torch.empty(d, d, **bf).normal_(0.0, d ** -0.5)
    bqkv, bo = torch.zeros(3 * d, **bf), torch.zeros(d, **bf)
    Y, QKV, O = torch.empty(T, d, **bf), torch.empty(T, 3 * d, **bf), torch.empty(T, d, **bf)
    LSE = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.tpmlp_attention_workspace_size(S, B, H), dtype=torch.uint8, device="cuda")
    block = lambda: binding.tpmlp_attention_tp_forward(X, Wqkv, Wo, S, B, H, N, Y, bqkv=bqkv, bo=bo, causal=True,
                                                       QKV_out=QKV, O_out=O, LSE_out=LSE, ws=ws)
    # each call graph-timed after a settle pause (the rows before it leave the GPU at its power cap)
    ms_blk = time_graph(torch, block, 10)
    ms_core = time_graph(torch, lambda: binding.tpmlp_attention_core(QKV, S, B, H, O, causal=True, LSE=LSE), 10)
    # backward: the gradient of Y flows back through the block from the saved QKV, O and statistics
    dY = step.dY[:T] if getattr(step, "dY", None) is not None else torch.empty(T, d, **bf).normal_()
    dX, dWo, dQKV = torch.empty(T, d, **bf), torch.empty(d, d, **bf), torch.empty(T, 3 * d, **bf)
    dWqkv, dbqkv, dbo = torch.empty(d, 3 * d, **bf), torch.empty(3 * d, **bf), torch.empty(d, **bf)
    dO = torch.empty(T, d, **bf).normal_()
    wsb = torch.empty(binding.tpmlp_attention_backward_workspace_size(S, B, H), dtype=torch.uint8, device="cuda")
    ms_blk_b = time_graph(torch, lambda: binding.tpmlp_attention_tp_backward(
        X, Wqkv, Wo, QKV, O, LSE, dY, S, B, H, N, dX, dWqkv, dWo, dbqkv=dbqkv, dbo=dbo, causal=True, ws=wsb), 10)
    ms_core_b = time_graph(torch, lambda: binding.tpmlp_attention_core_backward(QKV, O, dO, LSE, S, B, H, dQKV,
                                                                                causal=True, ws=wsb), 10)
    core_flops = 4.0 * 128 * B * H * S * (S + 1) / 2          # Q K^T and P V over the visible (causal) pairs
    core_bwd_flops = 2.5 * core_flops                          # Q K^T, dO V^T, P^T dO, dS K, dS^T Q
    gemm_flops = 2.0 * T * d * 3 * d + 2.0 * T * d * d
    gemm_bwd_flops = 2.0 * gemm_flops                          # data and weight gradients of both projections
    peak = tensor_peak(pk, 0.0)[0]  # ten calls of each: the burst peak
    tf = lambda f, ms: round(f / (ms * 1e-3) / 1e12, 1)
    return {"workload": f"S={S} x B={B}, d={d}, {H} heads of 128 over N={N} shards, causal",
            "timing": "CUDA graph of 10 back-to-back calls after a settle pause; fractions of the burst peak",
            "block_ms": round(ms_blk, 4), "block_TFLOP/s": tf(core_flops + gemm_flops, ms_blk),
            "core_ms": round(ms_core, 4), "core_TFLOP/s": tf(core_flops, ms_core),
            "core_frac": round(core_flops / (ms_core * 1e-3) / 1e12 / peak, 3),
            "block_bwd_ms": round(ms_blk_b, 4), "block_bwd_TFLOP/s": tf(core_bwd_flops + gemm_bwd_flops, ms_blk_b),
            "core_bwd_ms": round(ms_core_b, 4), "core_bwd_TFLOP/s": tf(core_bwd_flops, ms_core_b),
            "core_bwd_frac": round(core_bwd_flops / (ms_core_b * 1e-3) / 1e12 / peak, 3)}


OTHER_ROWS = ("reduce_scatter_explicit", "rmsnorm_gather", "layernorm_gather_isolated", "layernorm_backward_isolated",
              "gemm2_bias_dropout_add",
              "dropout_backward", "layernorm_gather_long_sequence", "fp8", "attention_tp", "fp32_tiny_forward")


def run_other_rows(step, torch, binding, pk, only=None):
    """Rows of the hot path the step does not run: the explicit reduce-scatter (per-shard bf16 partials, then
    the reduce-scatter kernel), the RMS norm variant, the rest of the SP region, FP8, attention on the step's
    shapes, and the fp32 path on the tiny fp32 workload.  `only`: one name of OTHER_ROWS (the others are
    skipped)."""
    w = step.w
    out = {}
    want = lambda name: only is None or only == name
    if want("reduce_scatter_explicit") and w.sp and (w.F // w.N) % 64 == 0:
        P = torch.empty(w.N, w.T, w.d, dtype=torch.bfloat16, device="cuda")
        Yc = [torch.empty(w.T // w.N, w.d, dtype=torch.bfloat16, device="cuda") for _ in range(w.N)]
        g = 2.0 * w.T * w.d * w.F
        ms_p = time_calls(torch, lambda: binding.tpmlp_gemm2_partials(step.H, step.B, w.N, P), 10)
        rs = lambda: binding.tpmlp_reduce_scatter(P, w.N, Yc)
        ms_rs, ms_rs_e = time_graph(torch, rs, 20), time_calls(torch, rs, 20)
        rs_bytes = (w.N + 1) * w.T * w.d * 2.0
        out["gemm2_partials"] = {"ms": round(ms_p, 4), "TFLOP/s": round(g / (ms_p * 1e-3) / 1e12, 1),
                                 "frac": round(g / (ms_p * 1e-3) / 1e12 / tensor_peak(pk, 0.0)[0], 3)}
        out["reduce_scatter_explicit"] = hbm_row(rs_bytes, ms_rs, ms_rs_e, pk)
        del P, Yc
    if (want("rmsnorm_gather") or want("layernorm_gather_isolated") or want("layernorm_backward_isolated")) and \
            w.sp and w.backward:
        # the RMS norm variant of the gathered norm, and the LayerNorm beside it timed the same way; the calls
        # alternate between (X -> Xg) and (dY -> dXg) so each reads 2 T d bytes the previous call did not touch
        # (256 MB of inputs and outputs in all, about twice the L2)
        nb = 4.0 * w.T * w.d
        for name, fn in (("rmsnorm_gather", binding.tpmlp_rmsnorm_gather),
                         ("layernorm_gather_isolated", binding.tpmlp_layernorm_gather)):
            extra = (step.gamma,) if name.startswith("rms") else (step.gamma, step.beta)
            pair = lambda: (fn(step.Xc, *extra, w.N, step.Xg), fn(step.dYc, *extra, w.N, step.dXg))
            out[name] = hbm_row(nb, time_graph(torch, pair, 20) / 2.0, time_calls(torch, pair, 20) / 2.0, pk)
        # the LayerNorm backward alone, two sets of operands alternating (402 MB, three times the L2)
        nbb = 6.0 * w.T * w.d
        Xg2, dXc2 = torch.empty_like(step.Xg), [torch.empty_like(c) for c in step.dXc]
        Xg2.copy_(step.dXg)
        pair_b = lambda: (binding.tpmlp_layernorm_backward(step.Xc, step.gamma, step.dXg, w.N, step.dXc, step.dgamma,
                                                           step.dbeta, ws=step.lnws),
                          binding.tpmlp_layernorm_backward(step.dYc, step.gamma, Xg2, w.N, dXc2, step.dgamma,
                                                           step.dbeta, ws=step.lnws))
        out["layernorm_backward_isolated"] = hbm_row(nbb, time_graph(torch, pair_b, 10) / 2.0,
                                                     time_calls(torch, pair_b, 10) / 2.0, pk, launches=2)
        del Xg2, dXc2
        # the same bytes moved by a plain device copy (torch), timed the same way: what a launch of this size
        # reaches, beside the bandwidth peak measured on a 4 GB copy
        src_a, src_b = torch.empty_like(step.Xg), torch.empty_like(step.dXg)
        src_a.zero_(), src_b.zero_()
        cp = lambda: (step.Xg.copy_(src_a), step.dXg.copy_(src_b))
        out["copy_same_bytes"] = hbm_row(nb, time_graph(torch, cp, 20) / 2.0, time_calls(torch, cp, 20) / 2.0, pk,
                                         what="torch copy_ of one [T x d] bf16 tensor into another, alternating two "
                                              "pairs as the norm rows do")
        del src_a, src_b
    if (want("gemm2_bias_dropout_add") or want("dropout_backward")) and w.sp:
        # the rest of the sequence-parallel region on the step's shapes: the row-parallel GEMM with row bias,
        # dropout (p = 0.1) and residual in its chunked store, and the dropout backward (+ row-bias gradient)
        g = 2.0 * w.T * w.d * w.F
        b2 = step.gamma  # any [d] bf16 vector serves as the row bias here
        ms_t = time_calls(torch, lambda: binding.tpmlp_gemm2_bias_dropout_add(
            step.H, step.B, w.N, step.Yc, bias2=b2, p=0.1, seed=1, offset=2, R_chunks=step.Xc), 10)
        out["gemm2_bias_dropout_add"] = {"ms": round(ms_t, 4), "TFLOP/s": round(g / (ms_t * 1e-3) / 1e12, 1),
                                         "frac": round(g / (ms_t * 1e-3) / 1e12 / tensor_peak(pk, 0.0)[0], 3)}
        if w.backward:
            db2 = torch.empty(w.d, dtype=torch.bfloat16, device="cuda")
            dws = binding.workspace(binding.make_shape(w.T, w.d, w.F, w.N), binding.OP_DROPOUT_BWD)
            nb = 4.0 * w.T * w.d
            pair = lambda: (binding.tpmlp_dropout_backward(step.dYc, w.N, step.dXg, dbias2=db2, p=0.1, seed=1,
                                                           offset=2, ws=dws),
                            binding.tpmlp_dropout_backward(step.Yc, w.N, step.Xg, dbias2=db2, p=0.1, seed=1,
                                                           offset=3, ws=dws))
            ms_d = time_graph(torch, pair, 20) / 2.0
            # with the keep mask the forward saved (one bit per element, read instead of regenerated)
            masks = []
            for off in (2, 3):
                mk = torch.empty(binding.keep_mask_bytes(w.T, w.d), dtype=torch.uint8, device="cuda")
                binding.tpmlp_gemm2_bias_dropout_add(step.H, step.B, w.N, step.Yc, p=0.1, seed=1, offset=off,
                                                     keep_mask=mk)
                masks.append(mk)
            pair_m = lambda: (binding.tpmlp_dropout_backward(step.dYc, w.N, step.dXg, dbias2=db2, p=0.1, seed=1,
                                                             offset=2, ws=dws, keep_mask=masks[0]),
                              binding.tpmlp_dropout_backward(step.Yc, w.N, step.Xg, dbias2=db2, p=0.1, seed=1,
                                                             offset=3, ws=dws, keep_mask=masks[1]))
            nbm = nb + w.T * w.d / 8.0
            out["dropout_backward"] = hbm_row(nbm, time_graph(torch, pair_m, 20) / 2.0,
                                              time_calls(torch, pair_m, 20) / 2.0, pk, launches=2,
                                              keep_mask="saved by the forward",
                                              regenerated_mask_ms=round(ms_d, 4),
                                              regenerated_mask_frac=round(nb / (ms_d * 1e-3) / 1e9 / pk["hbm_gbs"], 3))
    if want("layernorm_gather_long_sequence") and w.sp and w.d in (1024, 2048, 4096):
        # the LayerNorm forward on a sequence 8x as long (same d): enough rows per warp for the persistent,
        # software-pipelined kernel, whose start-up the step's 8192 rows do not amortise
        Tl = 8 * w.T
        xl = [torch.empty(Tl, w.d, dtype=torch.bfloat16, device="cuda").normal_() for _ in range(2)]
        yl = [torch.empty(Tl, w.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        nb = 4.0 * Tl * w.d
        pair = lambda: [binding.tpmlp_layernorm_gather(list(xl[k].split(Tl // w.N)), step.gamma, step.beta, w.N, yl[k])
                        for k in range(2)]
        out["layernorm_gather_long_sequence"] = hbm_row(nb, time_graph(torch, pair, 10) / 2.0,
                                                        time_calls(torch, pair, 10) / 2.0, pk, tokens=Tl)
        del xl, yl
    if want("fp8") and (w.sp and w.backward and w.T % 16 == 0 and w.d % 16 == 0 and w.F % 16 == 0 and
            w.d in (256, 512, 1024, 2048, 4096, 8192)):
        out["fp8"] = run_fp8_step(step, torch, binding, pk)
    if want("attention_tp") and w.d % 128 == 0 and w.T % 2 == 0:
        out["attention_tp"] = run_attention(step, torch, binding, pk)
    if not want("fp32_tiny_forward"):
        return out
    t = inputs.WORKLOADS["tiny_fp32_fwd"]
    f32 = lambda name: torch.from_numpy(np.ascontiguousarray(inputs.draw(t, name)[0])).cuda()
    X, A, B, b = f32("X"), f32("A"), f32("B"), f32("bias")
    Y = torch.empty(t.T, t.d, dtype=torch.float32, device="cuda")
    ws = binding.workspace(binding.make_shape(t.T, t.d, t.F, t.N, binding.FP32), binding.OP_FWD)
    ms = time_calls(torch, lambda: binding.tpmlp_forward(X, A, B, b, t.N, Y, ws=ws), 200)
    out["fp32_tiny_forward"] = {"us": round(ms * 1e3, 2), "GFLOP/s": round(4.0 * t.T * t.d * t.F / (ms * 1e-3) / 1e9, 1),
                                "workload": t.name, "bound": "launch latency (2 launches of a few CTAs)"}
    return out


class nvtx_range:
    """An NVTX range around a bench phase (visible to profilers; no effect on the timing)."""

    def __init__(self, torch, name):
        self.torch, self.name = torch, name

    def __enter__(self):
        self.torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        self.torch.cuda.nvtx.range_pop()


def timed_passes(step, torch, steps, gpu_index, barrier=lambda: None):
    """Time `steps` back-to-back steps with an event at every step boundary (the step's kernels follow one
    another with nothing between them), then, after a pause, the same number of steps with an event between
    consecutive kernels for the per-kernel breakdown.  SM clocks are sampled throughout."""
    nseg = len(step.kernels())
    ev = lambda: torch.cuda.Event(enable_timing=True)
    step_ev = [ev() for _ in range(steps + 1)]
    seg_ev = [[ev() for _ in range(nseg + 1)] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clk:
        time.sleep(0.3)
        t0 = time.perf_counter()
        e0 = time.time()
        with nvtx_range(torch, f"{step.w.name}: {steps} timed steps"):
            step_ev[0].record()
            for k in range(steps):
                step.run()
                step_ev[k + 1].record()
            torch.cuda.synchronize()
        e1 = time.time()
        wall = time.perf_counter() - t0
        time.sleep(1.0)  # the clocks recover from the timed steps' load before the breakdown
        b0 = time.time()
        with nvtx_range(torch, f"{step.w.name}: per-kernel breakdown"):
            for k in range(steps):
                step.run(seg_ev[k])
            torch.cuda.synchronize()
        b1 = time.time()
        time.sleep(0.15)
    barrier()
    step_ms = [step_ev[k].elapsed_time(step_ev[k + 1]) for k in range(steps)]
    seg_ms = [sum(seg_ev[k][i].elapsed_time(seg_ev[k][i + 1]) for k in range(steps)) / steps for i in range(nseg)]
    return {"step_ms": step_ms, "total_ms": step_ev[0].elapsed_time(step_ev[steps]), "seg_ms": seg_ms,
            "clocks": clk.summary(e0, e1), "clocks_breakdown": clk.summary(b0, b1), "wall": wall}


def kernel_table(step, seg_ms, pk, region_s, sm_count, sm_mhz, workload_key):
    """Per-segment rates: GEMMs in TFLOP/s against the tensor peak that fits the region's length and against
    the peak at the clock the run held; row kernels in GB/s of algorithmic bytes against measured HBM.  Also
    the dominant (longest) GEMM: (name, ms, flops, TFLOP/s, peak, peak kind, clock peak)."""
    peak, kind = tensor_peak(pk, region_s)
    cpk = clock_peak(sm_count, sm_mhz)
    kern, dom = {}, None
    for (name, nl, work, unit), avg in zip(step.kernels(), seg_ms):
        if unit == "F":
            ach = work / (avg * 1e-3) / 1e12
            kern[name] = {"ms": round(avg, 4), "TFLOP/s": round(ach, 1), "frac": round(ach / peak, 3),
                          "frac_clock": round(ach / cpk, 3) if cpk else None,
                          "dram_bytes": measured_traffic(name, workload_key)}
            if dom is None or avg > dom[1]:
                dom = (name, avg, work, ach, peak, kind, cpk)
        else:
            ach = work / (avg * 1e-3) / 1e9
            kern[name] = {"ms": round(avg, 4), "GB/s": round(ach, 1), "frac": round(ach / pk["hbm_gbs"], 3),
                          "launches": nl, "dram_bytes": measured_traffic(name, workload_key)}
    return kern, dom


FORWARD_ROWS = ("mlp7b_fwd", "sp_large_fwd")


def run_forward_row(name, torch, binding, pk, gpu_index, steps=30, warmup=3):
    """A forward-only workload timed like the step: the 7B-shaped MLP forward (T = 8192, d = 4096,
    F = 16384) or the d = 8192 sequence-parallel forward (T = 4096 in 512-row chunks, F = 32768).  Inputs are
    drawn on the device with torch's seeded generator, the workload's distributions."""
    w = inputs.WORKLOADS[name]
    step = Step(w, torch, binding, seed=0, on_device=True)
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    r = timed_passes(step, torch, steps, gpu_index)
    sms = torch.cuda.get_device_properties(gpu_index).multi_processor_count
    region_s = r["total_ms"] * 1e-3
    kern, dom = kernel_table(step, r["seg_ms"], pk, region_s, sms, r["clocks_breakdown"].get("sm_mhz"), w.name)
    flops = useful_flops(w)
    ms = r["total_ms"] / steps
    peak, kind = tensor_peak(pk, region_s)
    cpk = clock_peak(sms, r["clocks"].get("sm_mhz"))
    ach = flops / (ms * 1e-3) / 1e12
    ln = None
    if w.sp:
        # the gathered LayerNorm alone at this shape, two buffer sets alternating, in a CUDA graph
        X2, Xg2 = torch.empty_like(step.X).normal_(), torch.empty_like(step.Xg)
        X2c = list(X2.split(step.rows))
        pair = lambda: (binding.tpmlp_layernorm_gather(step.Xc, step.gamma, step.beta, w.N, step.Xg),
                        binding.tpmlp_layernorm_gather(X2c, step.gamma, step.beta, w.N, Xg2))
        ln = hbm_row(4.0 * w.T * w.d, time_graph(torch, pair, 20) / 2.0, time_calls(torch, pair, 20) / 2.0, pk,
                     rows_per_chunk=step.rows)
        del X2, Xg2, X2c
    out = {"workload": f"{w.name}: T={w.T} ({w.batch} x {w.seq}), d={w.d}, F={w.F}, N={w.N}"
                       + (f", LayerNorm on {w.T // w.N}-row chunks" if w.sp else ""),
           "steps": steps, "ms_per_step": round(ms, 4), "step_ms": percentiles(r["step_ms"]),
           "TFLOP/s": round(ach, 1), "frac": round(ach / peak, 3), "peak_kind": f"measured bf16 {kind}",
           "frac_clock": round(ach / cpk, 3) if cpk else None, "tokens_per_s": round(w.T / (ms * 1e-3), 1),
           "kernels": kern, "clocks": r["clocks"], "inputs": "torch seeded device generator, the recipe's "
                                                            "distributions"}
    if ln is not None:
        out["layernorm_gather_isolated"] = ln
    del step
    torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch

    from tensor_transformer_mlp_tp_gb300 import binding, build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(binding.lib_path()):
        build.build()
    if dist is not None:
        dist.barrier()
    binding.lib()

    step = Step(w, torch, binding)
    sms = torch.cuda.get_device_properties(local).multi_processor_count

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    st, site = binding.tpmlp_get_device_status()
    if st != binding.OK:
        raise RuntimeError(f"device status after warm-up: {binding.status_string(st)} (site {site})")

    r = timed_passes(step, torch, args.steps, local, barrier=(dist.barrier if dist is not None else lambda: None))
    total_ms = max_over_ranks(r["total_ms"], dist)
    st, site = binding.tpmlp_get_device_status()
    if st != binding.OK:
        raise RuntimeError(f"device status after timing: {binding.status_string(st)} (site {site})")

    pk, pk_kind = peaks()
    flops = useful_flops(w)
    value = whole_job_rate(flops, args.steps, world, total_ms) / 1e12
    tokens_per_s = whole_job_rate(w.T, args.steps, world, total_ms)
    clocks = r["clocks"]
    region_s = r["total_ms"] * 1e-3
    kern, dom = kernel_table(step, r["seg_ms"], pk, region_s, sms, r["clocks_breakdown"].get("sm_mhz"), w.name)

    if args.step_only:
        # profiling runs: the timed step and its breakdown only
        args.only_row, args.no_forward_rows, args.no_cpu_baseline = "none", True, True
    if args.only_row is None:
        with nvtx_range(torch, "e2e through the block calls"):
            e2e_ms, h2d, d2h = run_e2e(step, args, torch, binding)
        st, site = binding.tpmlp_get_device_status()
        if st != binding.OK:
            raise RuntimeError(f"device status after e2e: {binding.status_string(st)} (site {site})")
        e2e_ms = max_over_ranks(e2e_ms, dist)
    with nvtx_range(torch, "other rows"):
        other = run_other_rows(step, torch, binding, pk, only=args.only_row) if args.only_row != "none" else {}
    st, site = binding.tpmlp_get_device_status()
    if st != binding.OK:
        raise RuntimeError(f"device status after the other rows: {binding.status_string(st)} (site {site})")
    if world == 1 and not args.no_forward_rows:
        # the forward-only workloads that carry the d = 4096 / 8192 forward GEMM rates and the LayerNorm at
        # 512-row chunks; the step's buffers are released first (the d = 8192 weights take 1 GiB)
        keep = (w.name, w.T, w.d, w.F)
        del step
        torch.cuda.empty_cache()
        for name in FORWARD_ROWS:
            if (args.only_row is None or args.only_row == name) and name != keep[0]:
                with nvtx_range(torch, f"forward row {name}"):
                    other[name] = run_forward_row(name, torch, binding, pk, local)
        st, site = binding.tpmlp_get_device_status()
        if st != binding.OK:
            raise RuntimeError(f"device status after the forward rows: {binding.status_string(st)} (site {site})")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only_row is None:
        dt, tok, fl = oracle_sample(w, tokens=args.oracle_tokens)
        cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "tokens_per_s": tok / dt, "seconds": round(dt, 2),
               "sample": f"{tok} of {w.T} tokens through the fp64 oracle with the full d={w.d}, F={w.F} weights "
                         f"(numpy float64, BLAS matmul on {cores} threads)"}
    if rank != 0:
        dist.destroy_process_group() if dist is not None else None
        return
    launches = sum(n for _, n, _, _ in Step.kernels_of(w)) * args.steps
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(tokens_per_s, 1),
        "step_ms": percentiles(r["step_ms"]),
        "config": {"workload": w.name, "tokens": w.T, "batch": w.batch, "seq": w.seq, "d": w.d, "ffn": w.F,
                   "n_shards": w.N, "sequence_parallel": w.sp, "backward": w.backward,
                   "parallelism": f"tp{w.N} shards on one GPU" + (f", {world} replicas" if world > 1 else ""),
                   "l2": "inputs larger than L2 (weights alone 2 x d x F x 2 bytes)",
                   "host_wall_s": round(r["wall"], 3)},
        "roofline": {"bound": "tensor", "kernel": dom[0], "achieved": round(dom[3], 1), "peak": dom[4],
                     "unit": "TFLOP/s", "frac": round(dom[3] / dom[4], 3),
                     "traffic": measured_traffic(dom[0], w.name),
                     "peak_kind": f"{pk_kind} bf16 {dom[5]} (timed region {region_s:.3f} s; the sustained peak "
                                  f"from {SUSTAINED_AFTER_S:g} s)",
                     "clock_peak": round(dom[6], 1) if dom[6] else None,
                     "frac_clock": round(dom[3] / dom[6], 3) if dom[6] else None,
                     "clock_peak_kind": f"{BF16_FLOP_PER_CLK_SM:g} flop/clk/SM x {sms} SMs x the median SM clock "
                                        "sampled during the breakdown pass"},
        "kernels": kern,
        "e2e": {"value": round(whole_job_rate(flops, args.steps, world, e2e_ms * args.steps) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "what": e2e_what(w)}
               if args.only_row is None else {"skipped": "--step-only" if args.step_only else "--only-row " + args.only_row},
        "other_rows": other,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if args.cpu_baseline_configs and rank == 0 and world == 1:
        line["cpu_baseline_configs"] = cpu_baseline_configs()
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# The five configurations in their listed order.
CONFIGS = {1: "tiny_fp32_fwd", 2: "gpt2_medium_fwd", 3: "mlp7b_fwd", 4: "sp_block_fwd_bwd", 5: "sp_large_fwd"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sp_block_fwd_bwd", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--config", type=int, choices=sorted(CONFIGS), default=None,
                    help="select the workload by its number in the list of configurations (1 tiny fp32, 2 GPT-2-"
                         "medium, 3 7B, 4 SP block forward+backward, 5 d=8192 SP forward)")
    ap.add_argument("--oracle-tokens", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-configs", action="store_true",
                    help="also time the oracle on a 64-token sample of every configuration (the full tiny one) on "
                         "the host cores; minutes of host work for the weight draws")
    ap.add_argument("--step-only", action="store_true",
                    help="time the step and its per-kernel breakdown only (no e2e, other rows or CPU baseline): for "
                         "profiling")
    ap.add_argument("--no-forward-rows", action="store_true",
                    help="skip the forward-only 7B and d=8192 rows timed after the step")
    ap.add_argument("--only-row", choices=OTHER_ROWS + FORWARD_ROWS, default=None,
                    help="after the step, time only this row of other_rows (no e2e, no CPU baseline): for profiling")
    args = ap.parse_args()
    if args.config is not None:
        args.workload = CONFIGS[args.config]
    w = inputs.WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("bench.py times the bf16 workloads; the fp32 configuration (tiny_fp32_fwd) is the "
                         "other_rows.fp32_tiny_forward row of every run")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
