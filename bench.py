"""Throughput of the tensor-parallel hot path on one GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * the sharded MLP block at the 8.3B-layer shape (T = 4096 tokens, h = 3072,
    f = 12288, t = 8 shards): mp_mlp_fwd_fused (column-parallel GEMM + GeLU and
    row-parallel GEMM with the shard sum, one launch) then mp_mlp_bwd_fused (dU
    with GeLU', dX with the shard sum, dA, dB, one launch);
  * the vocab-parallel fused output GEMM + cross-entropy at the 1.2B-model
    shape (T = 8192, h = 1536, vocabulary 50,257 padded to 51,200, t = 8):
    mp_vocab_ce_partials then mp_vocab_ce_combine.

value = algorithmic FLOP of the step (12 T h f for the MLP, 2 T h v_pad for the
logits) / device time, in TFLOP/s. Inputs are resident in HBM when the timed
region starts; L2 is flushed (256 MiB write) between timed steps, outside the
per-step CUDA events. `e2e` repeats the step through the same C-ABI calls with
pinned HOST buffers, the host-to-device copies of the inputs and the
device-to-host copies of the results inside the timed region.

Beside the timed steps (never inside `value`): `sustained` runs the same step back
to back for several seconds, long enough for the board's power cap to set the
clock, with the SM clock sampled and each chunk of steps binned by the clock it
ran at; `ce_8p3b` times the fused cross-entropy at the 8.3B-layer width (T = 4096,
h = 3072, the same vocabulary and t = 8) with its own roofline entry.

`--impl reference` times the float64 CPU oracle on bounded token samples of the
same workload instead (the reference arm); `cpu_baseline` in the main line is
the same oracle timed once on a bounded sample.

Multi-GPU (torchrun, N > 1): every rank runs its own replica of the step on
its own batch (no data-path collective); the time is the max over ranks and
value sums the ranks' work (weak scaling).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TFLOP/s and % of GB300 BF16 tensor peak: sharded MLP fwd+bwd; vocab-CE tokens/s"
MLP = dict(T=4096, h=3072, f=12288, t=8, seed=1003)
CE = dict(T=8192, h=1536, v_pad=51200, v_valid=50257, t=8, seed=1002)
CE_8P3B = dict(T=4096, h=3072, v_pad=51200, v_valid=50257, t=8, seed=1006)
SUSTAINED_S = 4.0     # seconds of back-to-back steps in the sustained leg
SUSTAINED_CHUNK = 50  # steps between the sustained leg's CUDA events
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS_PER_STEP = 4  # MLP fwd: 1, MLP bwd: 1, CE: 2
# Sources whose hash a committed ncu summary records, per kernel: its DRAM counters are reported only
# while they still describe the code that runs.
CE_SOURCES = ("mptp_gemm.cuh", "mptp_ptx.cuh", "mptp_launch.cuh", "mptp_ce.cu")
CHAIN_SOURCES = ("mptp_gemm_chain.cuh", "mptp_gemm.cuh", "mptp_ptx.cuh", "mptp_launch.cuh", "mptp_mlp_fused.cu")


def mlp_flop(w=MLP):
    return 12.0 * w["T"] * w["h"] * w["f"]


def ce_flop(w=CE):
    return 2.0 * w["T"] * w["h"] * w["v_pad"]


def step_flop():
    return mlp_flop() + ce_flop()


# Dense bf16 tensor-core rate of one sm_103 SM (tcgen05 kind::f16, FLOP per clock).
BF16_FLOP_PER_CLK_PER_SM = 8192


def peak_table(value, mlp_tf, ce_tf, peaks, peak_src, dev, clocks):
    """Fractions of three denominators, as [step, MLP fwd+bwd, CE]: the theoretical dense bf16
    peak (SMs x per-SM rate x the SM clock: the maximum nvidia-smi reports, and the median it
    sampled during the timed steps), and the measured burst and sustained bf16 GEMM rates."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    mhz = (clocks or {}).get("sm_max_mhz")
    if not mhz:
        mhz = getattr(props, "clock_rate", 0) / 1000.0 or 2070.0
    med = (clocks or {}).get("sm_mhz") or mhz
    den = {"theoretical_max_clock": theoretical_tflops(dev, mhz), "theoretical_sampled_clock": theoretical_tflops(dev, med),
           "measured_burst": peaks["bf16_tflops"], "measured_sustained": peaks["bf16_tflops_sustained"]}
    out = {"tflops": den, "clock_mhz": {"max": mhz, "sampled_median": med}, "source": peak_src,
           "rate": f"{props.multi_processor_count} SMs x {BF16_FLOP_PER_CLK_PER_SM} FLOP/clk",
           "order": ["step", "mlp_fwd_bwd", "ce"]}
    out["frac"] = {k: [value / d, mlp_tf / d, ce_tf / d] for k, d in den.items()}
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(sources=CE_SOURCES):
    """sha256[:16] of the kernel sources with comments and blank lines removed, so that a
    recorded profile stays valid across comment-only edits."""
    import re
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "tensor_transformer_layer_gb300", "csrc", name)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(text.encode())
    return h.hexdigest()[:16]


def profiled_traffic(name="ce_logits_lse_ncu.txt", sources=CE_SOURCES):
    """DRAM bytes per launch of a kernel from its committed ncu summary, or None when
    the kernel sources changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as fh:
            kv = dict(line.split(":", 1) for line in fh if ":" in line and not line.startswith("#"))
    except OSError:
        return None
    kv = {k.strip(): v.strip() for k, v in kv.items()}
    if kv.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    try:
        return float(kv["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
def physical_gpu(local_rank: int) -> str:
    """nvidia-smi index (or UUID) of this rank's GPU, honouring CUDA_VISIBLE_DEVICES."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, timestamps: bool = False, period_ms: int = 50):
        self.gpu = gpu_index
        self.proc = None
        self.ts = timestamps
        self.period = period_ms
        self.text = ""

    def start(self):
        fields = ("timestamp," if self.ts else "") + self.FIELDS
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.text = out
        return summarize_clocks(out, timestamps=self.ts)


def parse_clock_rows(text: str, timestamps: bool = False):
    """(time or None, sm MHz, max MHz, watts, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap) per
    nvidia-smi sample; `time` is the sample's wall-clock time (epoch seconds) when the query
    led with the timestamp field."""
    import datetime
    rows = []
    off = 1 if timestamps else 0
    for r in csv.reader(io.StringIO(text)):
        r = [x.strip() for x in r]
        if len(r) < 9 + off:
            continue
        try:
            ts = None
            if timestamps:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            q = r[off:]
            rows.append((ts, float(q[1]), float(q[2]), float(q[3]), q[5], q[6], q[7], q[8]))
        except ValueError:
            continue
    return rows


def summarize_clocks(text: str, timestamps: bool = False):
    rows = [x[1:] for x in parse_clock_rows(text, timestamps)]
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    loaded = [x for x in rows if x[2] > 300.0] or rows  # samples drawing real power
    mhz = sorted(x[0] for x in loaded)
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    reasons = sorted({names[i] for x in loaded for i in range(4) if x[3 + i].lower() == "active"})
    return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(x[1] for x in rows), "reasons": reasons,
            "samples": len(loaded), "power_w_max": max(x[2] for x in rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
class Step:
    """Device buffers and the C-ABI calls of one step."""

    def __init__(self, dev, host_in=None):
        import torch

        import synth
        import tensor_transformer_layer_gb300 as mp
        self.mp = mp
        self.torch = torch
        self.dev = dev
        m, c = MLP, CE
        if host_in is None:
            mi = synth.mlp_inputs(m["T"], m["h"], m["f"], m["seed"])
            ci = synth.ce_inputs(c["T"], c["h"], c["v_pad"], c["v_valid"], c["seed"])
            host_in = {"X": mi["X"], "A": mi["A"], "B": mi["B"], "dZ": mi["dZ"], "Xc": ci["X"], "E": ci["E"],
                       "target": ci["target"]}
        self.host_in = host_in
        self.d = {k: v.to(dev) for k, v in self.host_in.items()}
        T, h, f = m["T"], m["h"], m["f"]
        bf = torch.bfloat16
        e = lambda *s, dt=bf: torch.empty(*s, dtype=dt, device=dev)
        self.d.update(Z=e(T, h), Y=e(T, f), U=e(T, f), dX=e(T, h), dA=e(h, f), dB=e(f, h), dU=e(T, f),
                      loss=e(c["T"], dt=torch.float32))
        self.ws = e(mp.mp_vocab_ce_workspace_bytes(c["T"], c["v_pad"], c["t"]), dt=torch.uint8)
        self.mlp_ws = mp.mp_mlp_fused_workspace(T, h, f, m["t"], device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out_names = ("Z", "dX", "dA", "dB", "loss")

    def twin(self):
        """Same host inputs, its own device buffers (for double-buffered pipelines)."""
        return Step(self.dev, host_in=self.host_in)

    def run(self, ev=None, stream=None):
        """One step on `stream` (default: the current stream). ev: optional dict of CUDA
        events to record around the MLP backward launch (b0, b1) and the CE logit kernel (ce0, ce1)."""
        mp, d = self.mp, self.d
        t = MLP["t"]
        kw = dict(d_status=self.status, stream=stream)
        mp.mp_mlp_fwd_fused(d["X"], d["A"], d["B"], d["Z"], d["Y"], d["U"], t=t, workspace=self.mlp_ws, **kw)
        if ev is not None:
            ev["b0"].record()
        mp.mp_mlp_bwd_fused(d["X"], d["A"], d["B"], d["U"], d["Y"], d["dZ"], d["dX"], d["dA"], d["dB"], d["dU"], t=t,
                            workspace=self.mlp_ws, **kw)
        if ev is not None:
            ev["b1"].record()
        if ev is not None:
            ev["ce0"].record()
        mp.mp_vocab_ce_partials(d["Xc"], d["E"], d["target"], self.ws, v_valid=CE["v_valid"], t=CE["t"], **kw)
        if ev is not None:
            ev["ce1"].record()
        mp.mp_vocab_ce_combine(self.ws, d["target"], d["loss"], v_pad=CE["v_pad"], v_valid=CE["v_valid"],
                               t=CE["t"], **kw)

    def check_status(self):
        s = int(self.status.item())
        if s != 0:
            raise RuntimeError(f"device status {s}: {self.mp.status_string(self.mp.mp_status_from_device(s))}")


def time_device(step, steps, warmup, flush):
    import torch
    for _ in range(warmup):
        step.run()
        flush.zero_()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        ev = {k: torch.cuda.Event(enable_timing=True) for k in ("s0", "s1", "b0", "b1", "ce0", "ce1")}
        ev["s0"].record()
        step.run(ev)
        ev["s1"].record()
        flush.zero_()
        evs.append(ev)
    torch.cuda.synchronize()
    step_ms = [e["s0"].elapsed_time(e["s1"]) for e in evs]
    ce_ms = [e["ce0"].elapsed_time(e["ce1"]) for e in evs]
    bwd_ms = [e["b0"].elapsed_time(e["b1"]) for e in evs]
    return step_ms, ce_ms, bwd_ms


def event_median(fn, reps, flush):
    """Median device time (ms) of fn() over `reps` calls, L2 flushed before each. All calls
    are enqueued before one synchronize, so the host's launch time of a short call is not
    counted as device time."""
    import torch
    evs = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) for a, b in evs)
    return ts[len(ts) // 2]


def time_breakdown(step, reps, flush):
    """Per-call device times (ms, median) of the step's four C-ABI calls, and of the MLP through the
    separate-launch entry points (mp_mlp_fwd / mp_mlp_bwd: the same outputs, bit for bit) for
    comparison."""
    import torch
    mp, d, t, ws = step.mp, step.d, MLP["t"], step.mlp_ws
    calls = {
        "mlp_fwd": lambda: mp.mp_mlp_fwd_fused(d["X"], d["A"], d["B"], d["Z"], d["Y"], d["U"], t=t, workspace=ws),
        "mlp_bwd": lambda: mp.mp_mlp_bwd_fused(d["X"], d["A"], d["B"], d["U"], d["Y"], d["dZ"], d["dX"], d["dA"],
                                               d["dB"], d["dU"], t=t, workspace=ws),
        "mlp_fwd_separate": lambda: mp.mp_mlp_fwd(d["X"], d["A"], d["B"], d["Z"], d["Y"], d["U"], t=t),
        "mlp_bwd_separate": lambda: mp.mp_mlp_bwd(d["X"], d["A"], d["B"], d["U"], d["Y"], d["dZ"], d["dX"], d["dA"],
                                                  d["dB"], d["dU"], t=t),
        "ce_partials": lambda: mp.mp_vocab_ce_partials(d["Xc"], d["E"], d["target"], step.ws,
                                                       v_valid=CE["v_valid"], t=CE["t"]),
        "ce_combine": lambda: mp.mp_vocab_ce_combine(step.ws, d["target"], d["loss"], v_pad=CE["v_pad"],
                                                     v_valid=CE["v_valid"], t=CE["t"]),
    }
    return {name: round(event_median(fn, reps, flush), 4) for name, fn in calls.items()}


def theoretical_tflops(dev, mhz):
    """Dense bf16 tensor peak at `mhz`: SMs x per-SM rate x clock."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    return props.multi_processor_count * BF16_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12


def bin_chunks_by_clock(chunk_windows, chunk_ms, chunk_flop, rows, bin_mhz=60.0):
    """Chunks of back-to-back steps binned by the SM clock they ran at.

    chunk_windows: (start, end) wall-clock seconds of each chunk; chunk_ms: its device time;
    rows: parsed nvidia-smi samples (time first). A chunk's clock is the median of the samples
    inside its window (chunks with none are left out). Returns one entry per clock bin, lowest
    first: the bin's centre, the chunks in it, their TFLOP/s and mean clock."""
    bins = {}
    for (a, b), ms in zip(chunk_windows, chunk_ms):
        mhz = sorted(x[1] for x in rows if x[0] is not None and a <= x[0] <= b and x[3] > 300.0)
        if not mhz or ms <= 0:
            continue
        c = mhz[len(mhz) // 2]
        k = round(c / bin_mhz) * bin_mhz
        e = bins.setdefault(k, {"ms": 0.0, "n": 0, "mhz": 0.0})
        e["ms"] += ms
        e["n"] += 1
        e["mhz"] += c
    return [{"mhz_bin": k, "chunks": e["n"], "mean_mhz": e["mhz"] / e["n"],
             "tflops": chunk_flop * e["n"] / (e["ms"] * 1e-3) / 1e12} for k, e in sorted(bins.items())]


def time_sustained(step, dev, gpu, seconds=SUSTAINED_S, chunk=SUSTAINED_CHUNK):
    """The step back to back for about `seconds` (no flush between steps, as in a training
    loop), long enough for the power cap to set the clock. CUDA events every `chunk` steps;
    the clock sampler's timestamps put each chunk at the clock it ran at."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(10):
        step.run()
    b.record()
    torch.cuda.synchronize()
    per_step = max(a.elapsed_time(b) / 10, 1e-3)
    n_chunks = max(4, int(seconds * 1e3 / (per_step * chunk)))
    sampler = ClockSampler(gpu, timestamps=True, period_ms=20)
    sampler.start()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_chunks + 1)]
    torch.cuda.synchronize()
    t0 = time.time()
    evs[0].record()
    for c in range(n_chunks):
        for _ in range(chunk):
            step.run()
        evs[c + 1].record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    step.check_status()
    ends = [evs[0].elapsed_time(e) for e in evs]
    chunk_ms = [ends[i + 1] - ends[i] for i in range(n_chunks)]
    windows = [(t0 + ends[i] * 1e-3, t0 + ends[i + 1] * 1e-3) for i in range(n_chunks)]
    rows = parse_clock_rows(sampler.text, timestamps=True)
    total_ms = ends[-1]
    steps = n_chunks * chunk
    ms_step = total_ms / steps
    tflops = step_flop() / (ms_step * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    mhz = clocks.get("sm_mhz")
    out = {"steps": steps, "seconds": total_ms * 1e-3, "ms_per_step": ms_step, "tflops": tflops,
           "peak": peaks["bf16_tflops_sustained"], "peak_source": f"{peak_src} bf16 sustained",
           "frac": tflops / peaks["bf16_tflops_sustained"],
           "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
           "by_clock": bin_chunks_by_clock(windows, chunk_ms, step_flop() * chunk, rows)}
    if mhz:
        theo = theoretical_tflops(dev, mhz)
        out["kcycles_per_step"] = ms_step * mhz  # time x median clock (ms x MHz = 1e3 cycles)
        out["theoretical_at_median_mhz"] = theo
        out["frac_of_theoretical_at_median_mhz"] = tflops / theo
    return out


def time_ce_8p3b(dev, reps, flush):
    """The fused cross-entropy at the 8.3B-layer width (T = 4096 = b 4 x s 1024, h = 3072,
    vocabulary 50,257 padded to 51,200, t = 8): the logit kernel (K6) alone, the whole call,
    and K6 against the burst bf16 peak (a kernel timed alone)."""
    import torch

    import synth
    import tensor_transformer_layer_gb300 as mp
    c = CE_8P3B
    ci = synth.ce_inputs(c["T"], c["h"], c["v_pad"], c["v_valid"], c["seed"])
    X, E, tg = ci["X"].to(dev), ci["E"].to(dev), ci["target"].to(dev)
    ws = torch.empty(mp.mp_vocab_ce_workspace_bytes(c["T"], c["v_pad"], c["t"]), dtype=torch.uint8, device=dev)
    loss = torch.empty(c["T"], dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    part = lambda: mp.mp_vocab_ce_partials(X, E, tg, ws, v_valid=c["v_valid"], t=c["t"], d_status=st)
    full = lambda: mp.mp_vocab_ce(X, E, tg, loss, ws, v_valid=c["v_valid"], t=c["t"], d_status=st)
    for _ in range(3):
        full()
    k6_ms = event_median(part, reps, flush)
    ce_ms = event_median(full, reps, flush)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())} in the 8.3B-layer cross-entropy")
    flop = 2.0 * c["T"] * c["h"] * c["v_pad"]
    peaks, peak_src = load_peaks()
    k6 = flop / (k6_ms * 1e-3) / 1e12
    out = {"T": c["T"], "h": c["h"], "v_pad": c["v_pad"], "v_valid": c["v_valid"], "t": c["t"],
           "ms": ce_ms, "tokens_per_s": c["T"] / (ce_ms * 1e-3), "tflops": flop / (ce_ms * 1e-3) / 1e12,
           "roofline": {"kernel": "K6 mp_vocab_ce_partials", "bound": "tensor", "achieved": k6,
                        "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": k6 / peaks["bf16_tflops"],
                        "peak_source": f"{peak_src} bf16 burst (kernel timed alone, L2 flushed, median of {reps})",
                        "traffic": profiled_traffic("ce_logits_lse_8p3b_ncu.txt"), "flop_per_launch": flop,
                        "avg_launch_ms": k6_ms}}
    del X, E, tg, ws, loss
    torch.cuda.empty_cache()
    return out


def rounded(obj, sig=5):
    """The same structure with floats rounded to `sig` significant digits (a shorter line)."""
    if isinstance(obj, float):
        if obj != obj or obj in (float("inf"), float("-inf")) or obj == 0.0:
            return obj
        return float(f"{obj:.{sig}g}")
    if isinstance(obj, dict):
        return {k: rounded(v, sig) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [rounded(v, sig) for v in obj]
    return obj


def combine_row(ms, peaks, peak_src):
    """The step's one memory-bound kernel, the cross-entropy combine (K7), against the measured
    HBM copy bandwidth. Algorithmic bytes: the (max, sum-exp) planes of every partition, one
    target logit, the target and the loss per token."""
    import tensor_transformer_layer_gb300 as mp
    T = CE["T"]
    P = mp.mp_vocab_ce_workspace_bytes(T, CE["v_pad"], CE["t"]) // (12 * T)
    nbytes = 8 * T * P + 12 * T
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "K7 mp_vocab_ce_combine", "bound": "hbm", "bytes": nbytes,
            "partitions": P, "ms": ms, "achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"],
            "frac": gbs / peaks["hbm_gbs"], "peak_source": peak_src,
            "timing": "one call after an L2 flush, launch included: latency-bound at a few MB"}


def time_next_rows(step, reps, flush):
    """Rows beyond the step (measured beside it, not inside `value`): the fused
    vocab-parallel cross-entropy backward on the step's CE workload."""
    import torch
    mp, d = step.mp, step.d
    T, h, v_pad, v_valid, t = CE["T"], CE["h"], CE["v_pad"], CE["v_valid"], CE["t"]
    dloss = torch.full((T,), 1.0 / T, dtype=torch.float32, device=d["Xc"].device)
    dXc = torch.empty(T, h, dtype=torch.bfloat16, device=d["Xc"].device)
    dE = torch.empty(v_pad, h, dtype=torch.bfloat16, device=d["Xc"].device)
    lse = torch.empty(T, dtype=torch.float32, device=d["Xc"].device)
    mp.mp_vocab_ce_lse(d["Xc"], d["E"], d["target"], d["loss"], lse, step.ws, v_valid=v_valid, t=t)
    # From the forward's exported log-sum-exp, in both workspace sizes: the minimum (one shard of
    # dZ at a time) and the one-pass size (every shard's dZ: one GEMM of each kind); and from the
    # forward's loss (the log-sum-exp rebuilt first), one pass.
    ce_ms = {}
    for mode, size, from_lse in (("shard_by_shard", mp.mp_vocab_ce_bwd_workspace_bytes, True),
                                 ("one_pass", mp.mp_vocab_ce_bwd_workspace_bytes_one_pass, True),
                                 ("one_pass_from_loss", mp.mp_vocab_ce_bwd_workspace_bytes_one_pass, False)):
        wsb = torch.empty(size(T, h, v_pad, t), dtype=torch.uint8, device=d["Xc"].device)
        if from_lse:
            fn = lambda: mp.mp_vocab_ce_bwd_lse(d["Xc"], d["E"], d["target"], lse, dloss, dXc, dE, wsb,
                                                v_valid=v_valid, t=t, d_status=step.status)
        else:
            fn = lambda: mp.mp_vocab_ce_bwd(d["Xc"], d["E"], d["target"], d["loss"], dloss, dXc, dE, wsb,
                                            v_valid=v_valid, t=t, d_status=step.status)
        fn()
        ce_ms[mode] = event_median(fn, reps, flush)
        step.check_status()
        del wsb
    ms = ce_ms["one_pass"]
    # vocab-parallel input embedding of the same T tokens (ids = the targets)
    emb = torch.empty(T, h, dtype=torch.bfloat16, device=d["Xc"].device)
    efn = lambda: mp.mp_vocab_embed(d["target"], d["E"], emb, v_valid=v_valid, t=t, d_status=step.status)
    efn()
    ems = event_median(efn, reps, flush)
    ebytes = 2.0 * T * h * 2 + 4.0 * T   # read T rows of E, write T rows, read the ids
    # context: a plain device copy of the same T x h bf16 rows, timed the same way (a 50 MB
    # kernel is dominated by its ramp and by the flush's dirty lines written back under it)
    csrc_ = torch.empty(T, h, dtype=torch.bfloat16, device=d["Xc"].device)
    cdst = torch.empty_like(csrc_)
    cms = event_median(lambda: cdst.copy_(csrc_), reps, flush)
    del csrc_, cdst
    peaks, peak_src = load_peaks()
    embed = {"ms": ems, "gbs": ebytes / (ems * 1e-3) / 1e9, "bytes": ebytes,
             "frac_of_hbm": ebytes / (ems * 1e-3) / 1e9 / peaks["hbm_gbs"], "hbm_peak_source": peak_src,
             "torch_copy_same_bytes_ms": cms, "vs_torch_copy": cms / ems}
    # head-parallel causal attention block at the 8.3B-layer shape (b = 4, s = 1024, 32 heads of 96, t = 8)
    import synth
    ab, as_, ah, aheads, at = 4, 1024, MLP["h"], 32, MLP["t"]
    aT = ab * as_
    ax = synth.normal_bf16((aT, ah), 1.0, 1005).to(d["Xc"].device)
    awqkv = synth.normal_bf16((ah, 3 * ah), 0.02, 1006).to(d["Xc"].device)
    awo = synth.normal_bf16((ah, ah), 0.02, 1007).to(d["Xc"].device)
    aout = torch.empty(aT, ah, dtype=torch.bfloat16, device=d["Xc"].device)
    aqkv = torch.empty(aT, 3 * ah, dtype=torch.bfloat16, device=d["Xc"].device)
    ao = torch.empty(aT, ah, dtype=torch.bfloat16, device=d["Xc"].device)
    afn = lambda: mp.mp_attn_fwd(ax, awqkv, awo, aout, aqkv, ao, b=ab, s=as_, heads=aheads, t=at,
                                 d_status=step.status)
    afn()
    ams = event_median(afn, reps, flush)
    hd = ah // aheads
    attn_core = 4.0 * ab * aheads * hd * as_ * (as_ + 1) / 2     # QK^T and PV over the causal pairs
    attn_flop = 2.0 * aT * ah * 3 * ah + attn_core + 2.0 * aT * ah * ah
    attn = {"ms": ams, "tflops": attn_flop / (ams * 1e-3) / 1e12, "flop": attn_flop,
            "shape": [ab, as_, ah, aheads, hd, at],
            "flop_note": "shape b,s,h,heads,d,t; QKV 6Th^2 + causal 4*b*heads*d*s(s+1)/2 + out 2Th^2"}
    attn.update(time_torch_attn(ax, awqkv, awo, ab, as_, aheads, reps, flush, attn_flop))
    algo = 4.0 * T * h * v_pad      # dX = dZ E and dE = dZ^T X
    executed = 6.0 * T * h * v_pad  # plus the logit recompute (logits are never stored)
    return {"ce_bwd": {"ms": ms, "tflops_algorithmic": algo / (ms * 1e-3) / 1e12,
                       "tflops_executed": executed / (ms * 1e-3) / 1e12, "tokens_per_s": T / (ms * 1e-3),
                       "ms_shard_by_shard": ce_ms["shard_by_shard"], "ms_from_loss": ce_ms["one_pass_from_loss"],
                       "flop_note": "from the exported lse, one-pass workspace; algorithmic 4Thv (dX, dE), "
                                    "executed adds the 2Thv logit recompute"},
            "vocab_embed": embed,
            "attn_fwd": attn}


def time_torch_attn(X, Wqkv, Wo, b, s, heads, reps, flush, flop):
    """Context for the attention block (never part of `value`): the same block composed from
    PyTorch, X Wqkv and O Wo on cuBLAS and causal scaled_dot_product_attention on its cuDNN
    backend, on the same device tensors."""
    import torch
    import torch.nn.functional as F
    T, h = X.shape
    d = h // heads
    try:
        from torch.nn.attention import SDPBackend, sdpa_kernel

        def block():
            qkv = X @ Wqkv
            q, k, v = (qkv[:, i * h:(i + 1) * h].view(b, s, heads, d).transpose(1, 2) for i in range(3))
            with sdpa_kernel([SDPBackend.CUDNN_ATTENTION]):
                o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
            return o.transpose(1, 2).reshape(T, h) @ Wo
        block()
        ms = event_median(block, reps, flush)
    except Exception as exc:  # a PyTorch without the cuDNN attention backend
        return {"torch_block": "unavailable: " + str(exc).splitlines()[0][:100]}
    return {"torch_block_ms": ms, "torch_block_tflops": flop / (ms * 1e-3) / 1e12,
            "torch_block_note": "PyTorch: X@Wqkv, F.scaled_dot_product_attention(is_causal) on cuDNN, O@Wo"}


def time_torch_context(step, reps, flush):
    """The step's two parts as a plain PyTorch composition on cuBLAS, on the same device
    tensors, for context only (never part of `value`): Z = GeLU(X A) B, erf form, with its
    backward through autograd (dX, dA, dB), unsharded; and the unfused loss, logits = X E^T
    materialised, then fp32 cross-entropy over the valid vocabulary. Median of `reps`, L2
    flushed before each."""
    import torch
    import torch.nn.functional as F
    d = step.d
    X, A, B, dZ = d["X"], d["A"], d["B"], d["dZ"]
    Xc, E, tgt = d["Xc"], d["E"], d["target"].long()
    v_valid = CE["v_valid"]

    def mlp():
        Xr, Ar, Br = (t.detach().requires_grad_(True) for t in (X, A, B))
        Z = F.gelu(Xr @ Ar, approximate="none") @ Br
        Z.backward(dZ)

    def ce():
        logits = (Xc @ E.t())[:, :v_valid].float()
        return F.cross_entropy(logits, tgt, reduction="none")

    mlp()
    ce()
    mlp_ms, ce_ms = event_median(mlp, reps, flush), event_median(ce, reps, flush)
    torch.cuda.empty_cache()
    return {"mlp_fwd_bwd_ms": mlp_ms, "mlp_tflops": mlp_flop() / (mlp_ms * 1e-3) / 1e12,
            "ce_ms": ce_ms, "ce_tflops": ce_flop() / (ce_ms * 1e-3) / 1e12,
            "note": "PyTorch/cuBLAS: F.gelu(X@A)@B + autograd; fp32 (X@E^T)[:, :v_valid] + F.cross_entropy"}


# Per-step host traffic of the two end-to-end measurements. "batch": the weights A, B, E are
# model state, uploaded once; every step copies in its batch (X, the upstream gradient dZ,
# the loss inputs Xc and targets) and reads back the per-token loss. "all": every input
# and every result (Z, dX, dA, dB, loss) crosses the host link every step.
E2E_BATCH_IN = ("X", "dZ", "Xc", "target")
E2E_BATCH_OUT = ("loss",)


def time_e2e(step, steps, warmup, in_names=None, out_names=None):
    """The step through the same C-ABI calls with its inputs copied in from pinned host
    memory and its results copied back, all inside the timed region (by default every
    input and every result). Copies and compute run as a double-buffered pipeline on three
    streams: step i+1's inputs go in and step i-1's results come out while step i computes."""
    import torch
    in_names = tuple(step.host_in) if in_names is None else in_names
    out_names = step.out_names if out_names is None else out_names
    host_in = {k: step.host_in[k].pin_memory() for k in in_names}
    host_out = {k: torch.empty(step.d[k].shape, dtype=step.d[k].dtype).pin_memory() for k in out_names}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    sets = [step, step.twin()]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    cur = torch.cuda.current_stream()
    for e in ev_comp + ev_out:
        e.record(cur)

    def one(i):
        b = i % 2
        st = sets[b]
        s_in.wait_event(ev_comp[b])          # buffer set b's previous step no longer reads its inputs
        with torch.cuda.stream(s_in):
            for k, v in host_in.items():
                st.d[k].copy_(v, non_blocking=True)
        ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        s_comp.wait_event(ev_out[b])         # its previous results have been copied out
        st.run(stream=s_comp)
        ev_comp[b].record(s_comp)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            for k, v in host_out.items():
                v.copy_(st.d[k], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        one(i)
    s_in.wait_event(ev_out[0])
    s_in.wait_event(ev_out[1])
    b.record(s_in)
    torch.cuda.synchronize()
    for st in sets:
        st.check_status()
    return a.elapsed_time(b) / steps, h2d, d2h


# ---------------------------------------------------------------------------
# oracle on the host cores (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
class OracleSample:
    """The float64 oracle on token samples of the same workload (full weights)."""

    def __init__(self, mlp_tokens: int, ce_tokens: int):
        import synth
        m, c = MLP, CE
        mi = synth.mlp_inputs(m["T"], m["h"], m["f"], m["seed"])
        ci = synth.ce_inputs(c["T"], c["h"], c["v_pad"], c["v_valid"], c["seed"])
        f64 = synth.to_f64
        self.X = f64(mi["X"][:mlp_tokens])
        self.dZ = f64(mi["dZ"][:mlp_tokens])
        self.A = f64(mi["A"])
        self.B = f64(mi["B"])
        self.Xc = f64(ci["X"][:ce_tokens])
        self.E = f64(ci["E"])
        self.tgt = ci["target"][:ce_tokens].numpy()
        self.mlp_tokens, self.ce_tokens = mlp_tokens, ce_tokens

    def flop(self):
        return (12.0 * self.mlp_tokens * MLP["h"] * MLP["f"] + 2.0 * self.ce_tokens * CE["h"] * CE["v_pad"])

    def run(self):
        import oracle
        oracle.mlp_fwd(self.X, self.A, self.B)
        oracle.mlp_bwd(self.X, self.A, self.B, self.dZ)
        oracle.ce_loss(self.Xc, self.E, self.tgt, CE["v_valid"])


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(sample: OracleSample, min_seconds: float, max_reps: int):
    t0 = time.perf_counter()
    reps = 0
    while True:
        sample.run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return sample.flop() * reps / el / 1e12, el, reps


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    sample = OracleSample(mlp_tokens=8, ce_tokens=16)
    for _ in range(args.warmup):
        sample.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.run()
    el = time.perf_counter() - t0
    value = sample.flop() * args.steps / el / 1e12
    desc = (f"float64 oracle per step on {sample.mlp_tokens} MLP tokens (full 3072x12288 weights, fwd+bwd) "
            f"and {sample.ce_tokens} CE tokens (full 51,200x1536 embedding)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {
        "workload": "sharded MLP fwd+bwd at the 8.3B-layer shape + vocab-parallel fused CE at the 1.2B shape",
        "mlp": {"T": MLP["T"], "b": 4, "s": 1024, "h": MLP["h"], "f": MLP["f"], "t": MLP["t"]},
        "ce": {"T": CE["T"], "b": 8, "s": 1024, "h": CE["h"], "v_pad": CE["v_pad"], "v_valid": CE["v_valid"],
               "t": CE["t"]},
        "flop_per_step": step_flop(),
        "l2": "flushed between timed steps (256 MiB write outside the step events); step inputs > L2",
        "inputs": "seeded synthetic bf16: X, dZ ~ N(0,1); A, B, E ~ N(0, 0.02); targets uniform in [0, 50257)",
    }


# ---------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("mptp", "reference"), default="mptp")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer pass (profiling runs)")
    ap.add_argument("--no-next-rows", action="store_true", help="skip the rows measured beside the step")
    ap.add_argument("--no-sustained", action="store_true", help="skip the seconds-long back-to-back leg")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the PyTorch/cuBLAS composition timed beside the step for context")
    ap.add_argument("--sweep", action="store_true",
                    help="time MLP fwd+bwd and the fused CE at every point of the layer sweep (one JSON line each)")
    ap.add_argument("--profile-case", choices=("none", "ce", "ce_full", "ce_8p3b", "ce_bwd", "mlp", "mlp_small",
                                               "mlp_split", "mlp_chain", "mlp_chain_small", "attn"),
                    default="none",
                    help="run only a small case of one entry point a few times (for ncu), print nothing")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.profile_case == "none":
        ap.error("--warmup must be >= 3")

    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)

    from tensor_transformer_layer_gb300 import build as _build
    # One rank compiles (when the library is missing or stale); the others wait, then load it.
    if rank == 0:
        _build.build()
    barrier(world)
    if rank != 0:
        _build.build()

    if args.profile_case != "none":
        return profile_case(args.profile_case, dev)
    if args.sweep:
        sampler = ClockSampler(physical_gpu(local_rank))
        sampler.start()
        rc = run_sweep(dev, max(args.steps // 20, 5), args.warmup)
        print(json.dumps({"sweep_clocks": sampler.stop()}), flush=True)
        return rc

    step = Step(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    step.run()
    torch.cuda.synchronize()
    step.check_status()

    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(physical_gpu(local_rank))
    sampler.start()
    step_ms, ce_ms, bwd_ms = time_device(step, args.steps, args.warmup, flush)
    clocks = sampler.stop()
    torch.cuda.synchronize()
    barrier(world)
    step.check_status()

    local_total = sum(step_ms)
    total_ms = max_over_ranks(local_total, world, dev)
    ms_per_step = total_ms / args.steps
    value = world * step_flop() * args.steps / (total_ms * 1e-3) / 1e12

    # The end-to-end leg right after the device-timed steps, in the same thermal state.
    e2e = e2e_all = None
    if not args.no_e2e:
        pipe = "double-buffered: H2D of step i+1 and D2H of step i-1 overlap step i's compute"
        e2e_ms, h2d, d2h = time_e2e(step, max(3, min(args.steps, 30)), 3, E2E_BATCH_IN, E2E_BATCH_OUT)
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        e2e = {"value": world * step_flop() / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "host_in": list(E2E_BATCH_IN), "host_out": list(E2E_BATCH_OUT),
               "resident": "weights A, B, E uploaded once (model state)", "pipeline": pipe}
        all_ms, h2d, d2h = time_e2e(step, max(3, min(args.steps, 30)), 3)
        all_ms = max_over_ranks(all_ms, world, dev)
        e2e_all = {"value": world * step_flop() / (all_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "ms_per_step": all_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    breakdown = time_breakdown(step, 9, flush)
    next_rows = None if args.no_next_rows else time_next_rows(step, 9, flush)
    context = None if args.no_context else time_torch_context(step, 9, flush)
    peaks, peak_src = load_peaks()
    ce_avg_ms = sum(ce_ms) / len(ce_ms)
    ce_achieved = ce_flop() / (ce_avg_ms * 1e-3) / 1e12
    traffic = profiled_traffic()
    bwd_avg_ms = sum(bwd_ms) / len(bwd_ms)
    bwd_flop = 8.0 * MLP["T"] * MLP["h"] * MLP["f"]   # dU, dX, dA, dB: four 2 T h f products
    bwd_achieved = bwd_flop / (bwd_avg_ms * 1e-3) / 1e12
    mlp_ms = breakdown["mlp_fwd"] + breakdown["mlp_bwd"]
    ce_call_ms = breakdown["ce_partials"] + breakdown["ce_combine"]

    step.check_status()
    sustained = None if args.no_sustained else time_sustained(step, dev, physical_gpu(local_rank))
    ce83 = None if args.no_next_rows else time_ce_8p3b(dev, 9, flush)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del step
        torch.cuda.empty_cache()
        sample = OracleSample(mlp_tokens=64, ce_tokens=128)
        v, el, reps = time_oracle(sample, min_seconds=10.0, max_reps=50)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"float64 oracle, {reps} pass(es) of {sample.mlp_tokens} MLP tokens (fwd+bwd, full "
                         f"weights) + {sample.ce_tokens} CE tokens (full embedding) in {el:.1f} s"}

    if rank == 0:
        mlp_tf = mlp_flop() / (mlp_ms * 1e-3) / 1e12
        ce_tf = ce_flop() / (ce_call_ms * 1e-3) / 1e12
        theo_sampled = theoretical_tflops(dev, clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0)
        # Contract keys first; the context objects next; the headline sub-metrics last, so that a
        # reader of only the line's tail still sees them.
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(),
            "gpu_launches": KERNELS_PER_STEP * (args.steps),
            "clocks": clocks,
            "roofline": {"kernel": "MLP backward in one launch (gemm_chain_kernel: K3 dU with GeLU', K4 dX with the "
                                   "f sum, K5a dA, K5b dB), the step's longest kernel", "bound": "tensor",
                         "achieved": bwd_achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": bwd_achieved / peaks["bf16_tflops"],
                         "peak_source": f"{peak_src} bf16 burst (timed inside short steps)",
                         "traffic": profiled_traffic("mlp_chain_8p3b_ncu.txt", CHAIN_SOURCES),
                         "algorithmic_flop_per_launch": bwd_flop, "avg_launch_ms": bwd_avg_ms,
                         "theoretical_at_sampled_clock": theo_sampled,
                         "frac_of_theoretical_at_sampled_clock": bwd_achieved / theo_sampled},
            "roofline_ce": {"kernel": "K6 mp_vocab_ce_partials (logit GEMM + online LSE epilogue)", "bound": "tensor",
                         "achieved": ce_achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": ce_achieved / peaks["bf16_tflops"],
                         "peak_source": f"{peak_src} bf16 burst (timed inside short steps)", "traffic": traffic,
                         "algorithmic_flop_per_launch": ce_flop(), "avg_launch_ms": ce_avg_ms,
                         "theoretical_at_sampled_clock": theo_sampled,
                         "frac_of_theoretical_at_sampled_clock": ce_achieved / theo_sampled},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "e2e_all_tensors": e2e_all,
            "torch_context": context,
            "memory_bound": combine_row(breakdown["ce_combine"], peaks, peak_src),
            "next_rows": next_rows,
            "pct_of_peak": peak_table(value, mlp_tf, ce_tf, peaks, peak_src, dev, clocks),
            "breakdown_ms": breakdown,
            "ce_8p3b": ce83,
            "sustained": sustained,
            "mlp_fwd_bwd_tflops": mlp_tf,
            "ce_tflops": ce_tf,
            "ce_tokens_per_s": CE["T"] / (ce_call_ms * 1e-3),
        }
        print(json.dumps(rounded(line)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_sweep(dev, reps, warmup):
    """MLP fwd+bwd and fused CE throughput at every sweep point: h in {1536, 1920, 2304,
    3072} (f = 4h), T in {2048, 8192}, t in {1, 2, 4, 8}, vocabulary 51,200 (50,257
    valid). Median of `reps` launches, L2 flushed before each. The MLP runs through the
    one-launch entry points; the separate-launch ones are timed beside them."""
    import torch

    import synth
    import tensor_transformer_layer_gb300 as mp
    peaks, peak_src = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def med(fn):
        for _ in range(warmup):
            fn()
        return event_median(fn, reps, flush)

    for h in (1536, 1920, 2304, 3072):
        f = 4 * h
        for T in (2048, 8192):
            mi = synth.mlp_inputs(T, h, f, seed=1004)
            d = {k: v.to(dev) for k, v in mi.items()}
            e = lambda *s_: torch.empty(*s_, dtype=torch.bfloat16, device=dev)
            Z, Y, U, dX, dA, dB, dU = e(T, h), e(T, f), e(T, f), e(T, h), e(h, f), e(f, h), e(T, f)
            ci = synth.ce_inputs(T, h, 51200, 50257, seed=1004)
            Xc, E, tg = ci["X"].to(dev), ci["E"].to(dev), ci["target"].to(dev)
            loss = torch.empty(T, dtype=torch.float32, device=dev)
            mws = mp.mp_mlp_fused_workspace(T, h, f, 8, device=dev)
            for t in (1, 2, 4, 8):
                ms = med(lambda: (mp.mp_mlp_fwd_fused(d["X"], d["A"], d["B"], Z, Y, U, t=t, workspace=mws),
                                  mp.mp_mlp_bwd_fused(d["X"], d["A"], d["B"], U, Y, d["dZ"], dX, dA, dB, dU, t=t,
                                                      workspace=mws)))
                sep_ms = med(lambda: (mp.mp_mlp_fwd(d["X"], d["A"], d["B"], Z, Y, U, t=t),
                                      mp.mp_mlp_bwd(d["X"], d["A"], d["B"], U, Y, d["dZ"], dX, dA, dB, dU, t=t)))
                ws = torch.empty(mp.mp_vocab_ce_workspace_bytes(T, 51200, t), dtype=torch.uint8, device=dev)
                ce_ms = med(lambda: mp.mp_vocab_ce(Xc, E, tg, loss, ws, v_valid=50257, t=t))
                mlp_tf = 12.0 * T * h * f / (ms * 1e-3) / 1e12
                ce_tf = 2.0 * T * h * 51200 / (ce_ms * 1e-3) / 1e12
                print(json.dumps({
                    "sweep": True, "h": h, "f": f, "T": T, "t": t, "heads": h // 96,
                    "mlp_fwd_bwd_ms": ms, "mlp_tflops": mlp_tf, "mlp_separate_ms": sep_ms,
                    "mlp_separate_tflops": 12.0 * T * h * f / (sep_ms * 1e-3) / 1e12,
                    "ce_ms": ce_ms, "ce_tflops": ce_tf, "ce_tokens_per_s": T / (ce_ms * 1e-3),
                    "pct_of_measured_bf16_sustained": {"mlp": mlp_tf / peaks["bf16_tflops_sustained"],
                                                       "ce": ce_tf / peaks["bf16_tflops_sustained"]},
                    "peak_source": peak_src}), flush=True)
            del d, Z, Y, U, dX, dA, dB, dU, Xc, E, tg, mws
            torch.cuda.empty_cache()
    return 0


def profile_case(which, dev):
    """Cases for ncu captures: 'ce' (T=2048), 'ce_8p3b' (T=4096, h=3072: 0.35 GB) and 'mlp' (the 8.3B
    layer, 0.7 GB) are small enough for multi-pass captures (under 1 GB on the device, 0.2-0.7 ms
    kernels, inputs > L2); 'mlp_small' is the sweep's T = 2048, h = 1536 point and 'mlp_split' its
    T = 2048, h = 3072 point (K2 on the split-K kernel); 'mlp_chain' and 'mlp_chain_small' run the
    one-launch forward and backward at the 8.3B layer and at T = 2048, h = 1536 (the other 'mlp'
    cases run the separate-launch kernels); 'ce_full' is the bench's CE launch, for
    one-pass metrics only; 'ce_bwd' is the CE backward on the bench's CE workload from the exported
    log-sum-exp, one call shard by shard and then one call in one pass (1.3 GB on the device; for
    the one-pass launch list)."""
    import torch

    import synth
    import tensor_transformer_layer_gb300 as mp
    if which == "attn":
        b, s_, h, heads, t = 4, 1024, MLP["h"], 32, MLP["t"]
        X = synth.normal_bf16((b * s_, h), 1.0, 1005).to(dev)
        Wqkv = synth.normal_bf16((h, 3 * h), 0.02, 1006).to(dev)
        Wo = synth.normal_bf16((h, h), 0.02, 1007).to(dev)
        e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=dev)
        out, QKV, O = e(b * s_, h), e(b * s_, 3 * h), e(b * s_, h)
        for _ in range(3):
            mp.mp_attn_fwd(X, Wqkv, Wo, out, QKV, O, b=b, s=s_, heads=heads, t=t)
        torch.cuda.synchronize()
        return 0
    if which == "ce_bwd":
        T, h, v_pad, v_valid, t = CE["T"], CE["h"], CE["v_pad"], CE["v_valid"], CE["t"]
        ci = synth.ce_inputs(T, h, v_pad, v_valid, seed=CE["seed"])
        X, E, tgt = ci["X"].to(dev), ci["E"].to(dev), ci["target"].to(dev)
        ws = torch.empty(mp.mp_vocab_ce_workspace_bytes(T, v_pad, t), dtype=torch.uint8, device=dev)
        loss = torch.empty(T, dtype=torch.float32, device=dev)
        lse = torch.empty_like(loss)
        mp.mp_vocab_ce_lse(X, E, tgt, loss, lse, ws, v_valid=v_valid, t=t)
        dl = torch.full((T,), 1.0 / T, dtype=torch.float32, device=dev)
        dX = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        dE = torch.empty(v_pad, h, dtype=torch.bfloat16, device=dev)
        for size in (mp.mp_vocab_ce_bwd_workspace_bytes, mp.mp_vocab_ce_bwd_workspace_bytes_one_pass):
            wsb = torch.empty(size(T, h, v_pad, t), dtype=torch.uint8, device=dev)
            mp.mp_vocab_ce_bwd_lse(X, E, tgt, lse, dl, dX, dE, wsb, v_valid=v_valid, t=t)
            torch.cuda.synchronize()
            del wsb
        return 0
    if which in ("ce", "ce_full", "ce_8p3b"):
        T, h, v_pad, v_valid, t = (2048 if which == "ce" else CE["T"]), 1536, 51200, 50257, 8
        seed = 1002
        if which == "ce_8p3b":
            T, h, seed = CE_8P3B["T"], CE_8P3B["h"], CE_8P3B["seed"]
        ci = synth.ce_inputs(T, h, v_pad, v_valid, seed=seed)
        X, E, tgt = ci["X"].to(dev), ci["E"].to(dev), ci["target"].to(dev)
        ws = torch.empty(mp.mp_vocab_ce_workspace_bytes(T, v_pad, t), dtype=torch.uint8, device=dev)
        loss = torch.empty(T, dtype=torch.float32, device=dev)
        for _ in range(3):
            mp.mp_vocab_ce(X, E, tgt, loss, ws, v_valid=v_valid, t=t)
    else:
        T, h, f, t = MLP["T"], MLP["h"], MLP["f"], MLP["t"]
        if which == "mlp_small":   # the sweep's smallest point: T = 2048, h = 1536
            T, h, f = 2048, 1536, 6144
        if which == "mlp_split":   # T = 2048, h = 3072: the row-parallel GEMM split over two pairs
            T, h, f = 2048, 3072, 12288
        if which == "mlp_chain_small":   # the one-launch forward and backward at T = 2048, h = 1536
            T, h, f = 2048, 1536, 6144
        mi = synth.mlp_inputs(T, h, f, seed=MLP["seed"])
        d = {k: v.to(dev) for k, v in mi.items()}
        e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=dev)
        Z, Y, U, dX, dA, dB, dU = e(T, h), e(T, f), e(T, f), e(T, h), e(h, f), e(f, h), e(T, f)
        ws = mp.mp_mlp_fused_workspace(T, h, f, t, device=dev)
        for _ in range(3):
            if which.startswith("mlp_chain"):
                mp.mp_mlp_fwd_fused(d["X"], d["A"], d["B"], Z, Y, U, t=t, workspace=ws)
                mp.mp_mlp_bwd_fused(d["X"], d["A"], d["B"], U, Y, d["dZ"], dX, dA, dB, dU, t=t, workspace=ws)
            else:
                mp.mp_mlp_fwd(d["X"], d["A"], d["B"], Z, Y, U, t=t)
                mp.mp_mlp_bwd(d["X"], d["A"], d["B"], U, Y, d["dZ"], dX, dA, dB, dU, t=t)
    torch.cuda.synchronize()
    return 0


if __name__ == "__main__":
    sys.exit(main())
