#!/usr/bin/env python3
"""Benchmark of the fused attention forward (and backward) on GB300.

One step = one fa_fwd launch over the whole workload (all B*H*N query rows),
inputs resident in HBM. Default workload: non-causal MHA, B=4 H=16 N=4096
d=128, fp16 in / fp16 out, fp32 accumulate, scale 1/sqrt(128).

Metric: attention forward TFLOPS = 4 B H N^2 d / time (halved for causal),
also reported as a percentage of 2.25 PFLOP/s dense fp16. With
--pass backward a step is one fa_bwd call (dQ, dK, dV from the forward's O
and LSE) and the metric is 10 B H N^2 d / time (the five N x N x d products
of the backward; halved for causal).

Prints ONE JSON line (rank 0). Besides the headline workload it times every
other named workload (the other 16-bit configurations and the two 8-bit
shapes) in the same process, with the same steps, warm-up, L2 flush and
untimed soak before the timed steps (--soak-s: every figure is taken at the
clock the board sustains under that load, which a 1.4 kW power cap sets),
under "other_workloads". The SM clock of each timed region is read from the kernels
themselves (clock64 / %globaltimer per CTA, fa_sm_clock_read), and the
clock-corrected tensor fraction FLOPs / (t x SMs x 8192 x f_clock) is reported
beside the fraction of the measured peak.

Reference arm (--impl reference): the fp64 CPU oracle timed on this host's
cores on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--pass forward|backward]
"""
from __future__ import annotations

import argparse
import hashlib
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

from attention_forward_flashattention_gb300 import inputs as I  # noqa: E402

DEFAULT_WORKLOAD = "mha_b4_h16_n4096_d128_fp16"
METRIC = "attention fwd TFLOPS (4BHN²d, causal halved) and % of 2.25 PF dense fp16"
METRIC_BWD = "attention bwd TFLOPS (10BHN²d, causal halved) and % of 2.25 PF dense fp16"
NOMINAL_DENSE_FP16_TFLOPS = 2250.0
# dense tensor-core FLOPs per SM per clock: a 128 x 128 x 16 16-bit tcgen05.mma
# (2 * 128 * 128 * 16 FLOPs) takes 64 cycles; 8-bit products run at twice that
TENSOR_FLOP_PER_CLK_SM = {"fp16": 8192.0, "bf16": 8192.0, "e4m3": 16384.0}
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=I.WORKLOAD_ORDER + list(I.FP8_WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "backward"],
                   help="backward: time fa_bwd (dQ, dK, dV) on a 16-bit workload")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--soak-s", type=float, default=1.5,
                   help="untimed loaded seconds before the timed steps (clock samples)")
    p.add_argument("--other-workloads", default="all", choices=["all", "none"],
                   help="also time every other named workload (same steps, warm-up, flush)")
    p.add_argument("--kernel", default="auto", choices=["auto", "one-cta", "pair"],
                   help="forward kernel of the headline: fa_fwd's own choice (auto), the "
                        "one-CTA kernel alone (through fa_fwd_noalloc) or fa_fwd_pair "
                        "(CTA pairs, head dimension 128)")
    return p.parse_args()


# ------------------------------------------------------------ helpers

def hbm_figure(plan, ms: float, peaks: dict) -> dict:
    """The step's algorithmic HBM bytes (inputs read once, outputs written
    once: the bytes the host path copies) over its time, against the measured
    copy bandwidth: the roofline of the small, latency-bound workloads, and
    context for the others."""
    nbytes = plan.h2d + plan.d2h
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    return {"bytes": nbytes, "gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
            "peak_source": "measured copy" if "hbm_gbs" in peaks else "fallback"}


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# the files fa_fwd_kernel (16-bit) is built and launched from
FWD_SOURCES = ("ptx.cuh", "fa_common.cuh", "fa_kernel.cuh", "fa_launch.cuh", "fa_fwd_d64.cu",
               "fa_fwd_d128.cu", "fa_host.cu")
# the files fa_fwd_pair_kernel is built and launched from
PAIR_SOURCES = ("ptx.cuh", "fa_common.cuh", "fa_kernel.cuh", "fa_pair.cuh", "fa_fwd_pair.cu",
                "fa_host.cu")
# the files the e4m3 instance of fa_fwd_kernel is built and launched from
FP8_SOURCES = ("ptx.cuh", "fa_common.cuh", "fa_kernel.cuh", "fa_launch.cuh", "fa_fwd_fp8.cu",
               "fa_host.cu")
KERNEL_SOURCES = {"one_cta": FWD_SOURCES, "pair": PAIR_SOURCES, "fp8": FP8_SOURCES}


def _code_only(text: str) -> str:
    """The source without // comments and blank lines (comment edits leave
    the compiled kernel, and so its traffic, unchanged)."""
    lines = []
    for ln in text.splitlines():
        code = ln.split("//", 1)[0].rstrip()
        if code.strip():
            lines.append(code)
    return "\n".join(lines)


def kernel_source_sha256(kind: str = "one_cta") -> str:
    """Hash of a forward kernel's source code (kind: the 16-bit one-CTA
    kernel, the CTA-pair kernel or the e4m3 kernel): a recorded DRAM traffic
    figure holds only for the code it was measured on."""
    from attention_forward_flashattention_gb300 import build as fabuild
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kind]):
        with open(os.path.join(fabuild.CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of the kernel that runs `workload` (entries named
    cta_pair:<workload> are the CTA-pair kernel's, *_e4m3 the 8-bit
    kernel's); else None. The file holds blocks: a kernel_source_sha256 line,
    then workload / dram_bytes_per_launch line pairs measured on those
    sources."""
    path = os.path.join(ROOT, "profiles", "fa_fwd_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    kind = ("pair" if workload.startswith(PAIR_PREFIX) else
            "fp8" if workload.endswith("_e4m3") else "one_cta")
    want = kernel_source_sha256(kind)
    cur_hash, cur_wl = None, None
    for ln in lines:
        if ":" not in ln or ln.lstrip().startswith("#"):
            continue
        k, v = (x.strip() for x in ln.split(":", 1))
        if k == "kernel_source_sha256":
            cur_hash = v
        elif k == "workload":
            cur_wl = v
        elif k == "dram_bytes_per_launch" and cur_wl == workload and cur_hash == want:
            return int(float(v))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        fd, self.path = tempfile.mkstemp(prefix="fa_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for ln in f:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(REASON_NAMES, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest `value` over all ranks (the slowest rank sets a job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, total_ms_max: float, steps: int, world: int) -> float:
    """Whole-job TFLOPS: every rank processes its own copy of the workload
    (weak scaling), so the job does world x flops per step in the slowest
    rank's time."""
    ms_per_step = total_ms_max / steps
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def oracle_sample_rows(w, nrows: int, seed: int) -> np.ndarray:
    """Rows of the workload for the CPU oracle: a few heads, rows spread over N."""
    rng = np.random.default_rng(seed)
    heads = sorted(set(rng.integers(0, w.B * w.H, size=4).tolist()))
    per = max(1, nrows // len(heads))
    rows = [h * w.N + int(i) for h in heads for i in rng.integers(0, w.N, size=per)]
    return np.array(sorted(rows), dtype=np.int64)


def sample_flops(w, rows: np.ndarray) -> float:
    """Metric FLOPs attributable to these rows: the workload's metric FLOPs per
    row (4 N d, halved for causal) times the number of rows."""
    return w.flops / (w.B * w.H * w.N) * len(rows)


def get_workload(name: str):
    return I.WORKLOADS[name] if name in I.WORKLOADS else I.FP8_WORKLOADS[name]


def workload_inputs(w):
    """Host inputs of w: (q, k, v) 16-bit values, or an I.Fp8Inputs for e4m3."""
    return I.fp8_inputs(w) if w.dtype == "e4m3" else I.qkv_bits(w)


def _gen_inputs(name: str):
    """Host inputs of a named workload (runs in a spawned worker process)."""
    return workload_inputs(get_workload(name))


def oracle_rows(w, x, rows):
    import oracle
    if w.dtype == "e4m3":
        return oracle.attn_fp8(x.q, x.k, x.vt, x.q_scale, x.k_scales, x.v_scale, w.causal,
                               w.scale, rows=rows)
    q, k, v = x
    return oracle.attn_rows(q, k, v, w.dtype, w.causal, w.scale, rows)


def time_oracle(w, x, target_s: float, seed: int, max_rows: int = 500_000):
    """Times the oracle on a row sample sized to about target_s seconds: a
    small calibration run, then sized runs (re-sized while the last one took
    under half the target, at most three times)."""
    import oracle
    cores = oracle.threads(0)
    n = 16 * cores
    rows = oracle_sample_rows(w, n, seed)
    t = time.perf_counter()
    oracle_rows(w, x, rows)
    dt = max(time.perf_counter() - t, 1e-3)
    for attempt in range(3):
        n = int(min(max(len(rows) * target_s / dt, len(rows)), max_rows))
        rows = oracle_sample_rows(w, n, seed + 1 + attempt)
        t = time.perf_counter()
        oracle_rows(w, x, rows)
        dt = time.perf_counter() - t
        if dt >= 0.5 * target_s or len(rows) >= max_rows:
            break
    return sample_flops(w, rows) / dt / 1e12, dt, len(rows), cores


# ------------------------------------------------------------ arms

def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    w = get_workload(args.workload)
    import oracle
    oracle.build()
    vals, secs = [], []
    if args.pass_ == "backward":
        # one step = the backward oracle on a few whole heads (about 12 s at N=4096)
        x, dob = I.qkv_bits(w), I.dout_bits(w)
        for s in range(args.warmup + args.steps):
            t = time.perf_counter()
            cpu = cpu_backward_sample(w, x, dob)
            if s >= args.warmup:
                vals.append(cpu["value"])
                secs.append(time.perf_counter() - t)
        metric, cores = METRIC_BWD, cpu["cores"]
        sample = cpu["sample"].split(",")[0] + " per step; TFLOPS = heads x (metric FLOPs per " \
                                               "head) / wall time"
    else:
        x = workload_inputs(w)
        step_target = 2.0
        nrows, cores = 0, oracle.threads(0)
        for s in range(args.warmup + args.steps):
            tf, dt, n, cores = time_oracle(w, x, step_target, seed=w.seed * 7 + s)
            if s >= args.warmup:
                vals.append(tf)
                secs.append(dt)
                nrows += n
        metric = METRIC
        sample = (f"{nrows // max(1, args.steps)} query rows per step (grouped over 4 heads) "
                  f"of {w.name}; TFLOPS = rows x (metric FLOPs per row) / wall time")
    value = statistics.mean(vals)
    ms = statistics.mean(secs) * 1e3
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, N(0,1))",
        "config": {**workload_config(w), "pass": args.pass_},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w) -> dict:
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
            "causal": w.causal, "scale": w.scale, "q_mult": w.q_mult,
            "global_batch": w.B, "seq_len": w.N}


class Plan:
    """What one timed step runs: `step()` on device-resident inputs, and
    `e2e_step()` with pinned host inputs copied in and results copied out."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def forward_plan(fa, torch, w, dev, stream, x=None, kernel="auto") -> Plan:
    """kernel: "auto" times fa_fwd (which picks the one-CTA or the CTA-pair
    kernel), "pair" fa_fwd_pair, "one_cta" the one-CTA kernel alone (through
    fa_fwd_noalloc, which always runs it)."""
    fp8 = w.dtype == "e4m3"
    x = workload_inputs(w) if x is None else x
    if fp8:
        # e4m3 codes (Q, K, V^T) and the per-block K scales; bf16 output
        tdt = torch.bfloat16
        host = [torch.from_numpy(np.ascontiguousarray(t)).pin_memory() for t in (x.q, x.k, x.vt)]
        host.append(torch.from_numpy(np.ascontiguousarray(x.k_scales)).pin_memory())
    else:
        tdt = torch.float16 if w.dtype == "fp16" else torch.bfloat16
        host = [torch.from_numpy(t.view(np.int16)).view(tdt).pin_memory() for t in x]
    dev_in = [h.to(dev) for h in host]
    o = torch.empty((w.B, w.H, w.N, w.d), dtype=tdt, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    oh = torch.empty(o.shape, dtype=tdt).pin_memory()
    lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    launch = fa.fa_query_launch(w.B, w.H, w.N, w.d, w.causal)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pair_units = w.B * w.H * ((w.N + 511) // 512)   # the pair kernel's 512-row units
    one_units = w.B * w.H * ((w.N + 255) // 256)    # the one-CTA kernel's 256-row units
    pair = kernel == "pair" or (kernel == "auto" and not fp8 and launch["cluster"] == 2)

    code = fa.FA_DTYPE_BF16 if w.dtype == "bf16" else fa.FA_DTYPE_FP16
    sh = int(stream.cuda_stream)

    def run(ins):
        if fp8:
            fa.attention_forward_fp8_into(ins[0], ins[1], ins[2], o, lse, x.q_scale, ins[3],
                                          x.v_scale, w.causal, w.scale, stream)
        elif kernel == "pair":
            fa.attention_forward_pair_into(ins[0], ins[1], ins[2], o, lse, w.causal, w.scale,
                                           stream)
        elif kernel == "one_cta":
            rc = fa.fa_fwd_noalloc(ins[0].data_ptr(), ins[1].data_ptr(), ins[2].data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N, w.d, w.causal,
                                   w.scale, code, sh)
            if rc != fa.FA_OK:
                raise fa.FaError(rc, "fa_fwd_noalloc")
        else:
            fa.attention_forward_into(ins[0], ins[1], ins[2], o, lse, w.causal, w.scale, stream)

    if fp8:
        e2e_path = "torch copies in, fa_fwd_fp8, copies out (one stream)"

        def e2e_step():
            run([h.to(dev, non_blocking=True) for h in host])
            oh.copy_(o, non_blocking=True)
            lh.copy_(lse, non_blocking=True)
    else:
        # the public host-buffer entry point: copies in / forward / copies out
        # overlapped over chunks of heads on three streams
        e2e_path = "fa_fwd_host (pinned host buffers, chunked copy / compute overlap)"
        ws = torch.empty(fa.fa_fwd_host_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                         device=dev)

        def e2e_step():
            fa.attention_forward_host_into(host[0], host[1], host[2], oh, lh, ws, w.causal,
                                           w.scale, stream)

    peak_note = ""
    if fp8:   # e4m3 dense rate is twice the 16-bit one (4.5 vs 2.25 PFLOP/s nominal)
        peak_note = " x 2 (e4m3 / bf16 nominal dense ratio)"
    return Plan(
        metric=METRIC, flops=w.flops, step=lambda: run(dev_in), e2e_step=e2e_step,
        e2e_path=e2e_path,
        h2d=sum(h.numel() * h.element_size() for h in host),
        d2h=o.numel() * o.element_size() + lse.numel() * 4,
        launches=1, peak_mult=2.0 if fp8 else 1.0, peak_note=peak_note,
        kernel=("fa_fwd_pair_kernel" if pair else "fa_fwd_kernel")
               + (" (fa_fwd's choice)" if kernel == "auto" and not fp8 else ""),
        launch_cfg=({"grid": 2 * min(pair_units, sms // 2), "threads": launch["threads"],
                     "cluster": 2, "units": pair_units} if pair else
                    {"grid": min(one_units, sms), "threads": launch["threads"],
                     "units": one_units} if launch["cluster"] == 2 else
                    {"grid": launch["grid"], "threads": launch["threads"],
                     "smem_bytes": None if fp8 else launch["smem_bytes"],
                     "units": launch["units"]}),
        traffic=recorded_traffic(PAIR_PREFIX + w.name if pair else w.name),
        cpu=lambda: cpu_forward_sample(w, x))


def cpu_forward_sample(w, x) -> dict:
    tf, dt, n, cores = time_oracle(w, x, target_s=12.0, seed=w.seed * 13)
    return {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": f"{n} query rows (grouped over 4 heads) of {w.name}, {dt:.1f} s wall; "
                      f"TFLOPS = rows x (metric FLOPs per row) / wall time"}


def backward_plan(fa, torch, w, dev, stream, x=None) -> Plan:
    if w.dtype not in ("fp16", "bf16"):
        raise SystemExit("--pass backward takes a 16-bit workload")
    tdt = torch.float16 if w.dtype == "fp16" else torch.bfloat16
    x = I.qkv_bits(w) if x is None else x
    dob = I.dout_bits(w)
    q, k, v, do = (torch.from_numpy(t.view(np.int16)).view(tdt).to(dev) for t in x + (dob,))
    # the forward's outputs feed the backward, as in training (computed once)
    o, lse = fa.attention_forward(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize(dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d) // 4, dtype=torch.float32,
                     device=dev)
    code = fa._dtype_code(q)
    sh = int(stream.cuda_stream)
    host = [t.cpu().pin_memory() for t in (q, k, v, o, lse, do)]
    outs_h = [torch.empty(q.shape, dtype=tdt).pin_memory() for _ in range(3)]

    def run(ins):
        rc = fa.fa_bwd(*(t.data_ptr() for t in ins[:3]), ins[3].data_ptr(), ins[5].data_ptr(),
                       ins[4].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       ws.data_ptr(), w.B, w.H, w.N, w.d, w.causal, w.scale, code, sh)
        if rc != fa.FA_OK:
            raise fa.FaError(rc, "fa_bwd")

    dev_in = [q, k, v, o, lse, do]

    def e2e_step():
        run([h.to(dev, non_blocking=True) for h in host])
        for hh, t in zip(outs_h, (dq, dk, dv)):
            hh.copy_(t, non_blocking=True)

    return Plan(
        metric=METRIC_BWD, flops=2.5 * w.flops, step=lambda: run(dev_in), e2e_step=e2e_step,
        e2e_path="torch copies in, fa_bwd, copies out (one stream)",
        h2d=sum(h.numel() * h.element_size() for h in host),
        d2h=3 * q.numel() * q.element_size(),
        launches=3, peak_mult=1.0, peak_note="",
        kernel="fa_bwd (D/LSE prep + fa_bwd_kernel dK,dV + fa_bwd_kernel dQ; whole call)",
        launch_cfg={"launches_per_step": 3, "workspace_bytes": ws.numel() * 4},
        traffic=None,
        cpu=lambda: cpu_backward_sample(w, x, dob))


def cpu_backward_sample(w, x, dob) -> dict:
    """The backward oracle on a few whole heads, one thread per head."""
    import oracle
    cores = oracle.threads(0)
    nh = max(1, min(cores, 4))
    heads = np.random.default_rng(w.seed * 17).choice(w.B * w.H, size=nh, replace=False)
    t = time.perf_counter()
    oracle.attn_bwd(*x, dob, w.dtype, w.causal, w.scale, heads=heads, nthreads=nh)
    dt = time.perf_counter() - t
    flops = 2.5 * w.flops / (w.B * w.H) * nh
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": nh, "kind": "oracle",
            "sample": f"{nh} whole heads of {w.name} (one thread each), {dt:.1f} s wall; "
                      f"TFLOPS = heads x (metric FLOPs per head) / wall time"}


def time_steps(fa, torch, plan, stream, dev, flush, steps: int, warmup: int, world: int,
               soak_s: float = 0.0, sampler_device=None) -> dict:
    """Warm-up, optional untimed soak (with nvidia-smi sampling), then `steps`
    timed steps between CUDA events on `stream`, L2 flushed before each.
    Returns the per-step times, the max-over-ranks total and the SM clock the
    kernels recorded during the timed steps."""
    import torch.distributed as dist
    sh = int(stream.cuda_stream)
    for _ in range(max(warmup, 3)):
        plan.step()
    rc = fa.fa_check(sh)
    if rc != fa.FA_OK:
        raise RuntimeError("warm-up failed: " + fa.status_string(rc))
    sampler = ClockSampler(sampler_device) if sampler_device is not None else None
    t_end = time.perf_counter() + soak_s
    while time.perf_counter() < t_end:   # untimed load so clock samples exist
        for _ in range(20):
            plan.step()
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    fa.fa_sm_clock_read(sh)              # clear: record only the timed launches
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()                    # evict L2 between steps (outside the events)
        starts[i].record(stream)
        plan.step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler is not None else None
    clk_mhz, ctas = fa.fa_sm_clock_read(sh)
    rc = fa.fa_check(sh)
    if rc != fa.FA_OK:
        raise RuntimeError("timed steps failed: " + fa.status_string(rc))
    times_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return {"times_ms": times_ms, "total_ms": max_over_ranks(sum(times_ms), world, dev),
            "clk64_mhz": clk_mhz if ctas > 0 else None, "ctas": ctas, "clocks": clocks}


def clock_corrected_frac(tflops: float, dtype: str, sms: int, mhz) -> float | None:
    """Achieved FLOP/s over the tensor cores' dense rate at the clock the
    kernels ran at: FLOPs / (t x SMs x FLOP/clk/SM x f_clock)."""
    if not mhz:
        return None
    return tflops * 1e12 / (sms * TENSOR_FLOP_PER_CLK_SM[dtype] * mhz * 1e6)


PAIR_PREFIX = "cta_pair:"   # other_workloads key: the CTA-pair kernel on a workload
ONE_PREFIX = "one_cta:"     # other_workloads key: the one-CTA kernel on a workload


def other_workload_names(headline: str, pass_: str, picks_pair=None) -> list[str]:
    """Every other named workload; in the forward pass also the 8-bit shapes
    and, on every head-dimension-128 16-bit workload (the headline's
    included), the kernel fa_fwd does not pick there, so both kernels are
    timed in the same run. picks_pair(name) says whether fa_fwd runs the
    CTA-pair kernel on a workload (default: on the non-causal ones)."""
    if picks_pair is None:
        picks_pair = lambda n: not I.WORKLOADS[n].causal  # noqa: E731
    names = [n for n in I.WORKLOAD_ORDER if n != headline]
    if pass_ == "forward":
        names += [n for n in I.FP8_WORKLOADS if n != headline]
        names += [(ONE_PREFIX if picks_pair(n) else PAIR_PREFIX) + n
                  for n in I.WORKLOAD_ORDER if I.WORKLOADS[n].d == 128]
    return names


def _base_name(name: str) -> str:
    return name.removeprefix(PAIR_PREFIX).removeprefix(ONE_PREFIX)


def run_ours(args, rank: int, world: int, local_rank: int):
    import concurrent.futures as cf
    import multiprocessing as mp

    # host inputs of the other workloads are generated by spawned workers
    # while the headline runs (spawned before any CUDA call)
    others = [] if args.other_workloads == "none" else other_workload_names(args.workload,
                                                                            args.pass_)
    pool = None
    futures = {}
    if others:
        pool = cf.ProcessPoolExecutor(max_workers=min(len(others), max(1, os.cpu_count() or 1)),
                                      mp_context=mp.get_context("spawn"))
        futures = {b: pool.submit(_gen_inputs, b)
                   for b in sorted({_base_name(n) for n in others}) if b != args.workload}

    import torch

    import attention_forward_flashattention_gb300 as fa
    from attention_forward_flashattention_gb300 import build as fabuild

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fabuild.build()
    fa.load_library()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if others:  # the other kernel of each head-dimension-128 workload, by fa_fwd's own choice
        others = other_workload_names(
            args.workload, args.pass_,
            picks_pair=lambda n: fa.fa_query_launch(*(getattr(I.WORKLOADS[n], k) for k in
                                                      ("B", "H", "N", "d", "causal")))["cluster"] == 2)
    w = get_workload(args.workload)
    stream = torch.cuda.current_stream(dev)
    make = backward_plan if args.pass_ == "backward" else forward_plan
    if args.kernel == "pair":
        if args.pass_ != "forward" or w.dtype == "e4m3" or w.d != 128:
            raise SystemExit("--kernel pair takes a 16-bit head-dimension-128 forward workload")
        plan = forward_plan(fa, torch, w, dev, stream, kernel="pair")
    elif args.kernel == "one-cta":
        if args.pass_ != "forward" or w.dtype == "e4m3":
            raise SystemExit("--kernel one-cta takes a 16-bit forward workload")
        plan = forward_plan(fa, torch, w, dev, stream, kernel="one_cta")
    else:
        plan = make(fa, torch, w, dev, stream)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    t = time_steps(fa, torch, plan, stream, dev, flush, args.steps, args.warmup, world,
                   soak_s=args.soak_s, sampler_device=local_rank)
    times_ms, total_ms = t["times_ms"], t["total_ms"]
    ms_per_step = total_ms / args.steps
    value = job_throughput(plan.flops, total_ms, args.steps, world)
    per_gpu_tflops = value / world

    # end to end through the public API: pinned host in, pinned host out
    e2e = None
    if not args.no_e2e:
        # the host-link figure is taken with the host quiet: the workers that
        # generate the other workloads' inputs (numpy, gigabytes written) finish
        # first, since they compete for host memory bandwidth and cores
        if futures:
            cf.wait(list(futures.values()))
        plan.e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            plan.e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        e2e = {"value": plan.flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": plan.h2d,
               "d2h_bytes_per_step": plan.d2h, "path": plan.e2e_path}

    peaks = measured_peaks()
    if "bf16_tflops" in peaks:
        peak16, peak_src = float(peaks["bf16_tflops"]), "measured bf16 burst (fp16 same nominal rate)"
    else:
        peak16, peak_src = FALLBACK_PEAK_TFLOPS, "fallback"

    # every other workload: same steps, warm-up, flush and untimed soak (so every
    # figure is taken at the clock the board sustains), one after another
    other = {}
    head_inputs = None
    for name in others:
        base = _base_name(name)
        ow = get_workload(base)
        if base in futures:
            x = futures[base].result()
        else:  # the headline workload on the pair kernel: its own inputs
            head_inputs = head_inputs if head_inputs is not None else workload_inputs(ow)
            x = head_inputs
        if name.startswith(PAIR_PREFIX):
            oplan = forward_plan(fa, torch, ow, dev, stream, x=x, kernel="pair")
        elif name.startswith(ONE_PREFIX):
            oplan = forward_plan(fa, torch, ow, dev, stream, x=x, kernel="one_cta")
        else:
            oplan = make(fa, torch, ow, dev, stream, x=x)
        ot = time_steps(fa, torch, oplan, stream, dev, flush, args.steps, args.warmup, world,
                        soak_s=args.soak_s)
        oms = ot["total_ms"] / args.steps
        otf = job_throughput(oplan.flops, ot["total_ms"], args.steps, world) / world
        opeak = oplan.peak_mult * peak16
        other[name] = {
            "value": otf * world, "unit": "TFLOPS", "ms_per_step": oms,
            "step_ms_median": statistics.median(ot["times_ms"]),
            "pct_of_2250_tflops": 100.0 * otf / NOMINAL_DENSE_FP16_TFLOPS,
            "frac": otf / opeak, "peak": opeak,
            "clk64_mhz": ot["clk64_mhz"],
            "clock_corrected_frac": clock_corrected_frac(otf, ow.dtype, sms, ot["clk64_mhz"]),
            "config": {k: v for k, v in workload_config(ow).items()
                       if k not in ("global_batch", "seq_len")},
            "kernel": oplan.kernel,
            "traffic": oplan.traffic,
            "hbm": hbm_figure(oplan, oms, peaks),
        }
        del oplan
        torch.cuda.empty_cache()
    if pool is not None:
        pool.shutdown()

    if rank != 0:
        return
    peak = plan.peak_mult * peak16
    peak_src = peak_src + plan.peak_note
    cpu = None if args.no_cpu_baseline else plan.cpu()
    line = {
        "metric": plan.metric, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded SplitMix64 + Box-Muller, N(0,1)), resident in HBM",
        "config": {**workload_config(w), "pass": args.pass_, "kernel": plan.kernel,
                   "parallelism": f"replicas x{world}",
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
                   **plan.launch_cfg},
        "pct_of_2250_tflops": 100.0 * per_gpu_tflops / NOMINAL_DENSE_FP16_TFLOPS,
        "roofline": {"bound": "tensor", "achieved": per_gpu_tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": per_gpu_tflops / peak,
                     "traffic": plan.traffic, "peak_source": peak_src,
                     "kernel": plan.kernel,
                     "clock_corrected_frac": clock_corrected_frac(per_gpu_tflops, w.dtype, sms,
                                                                  t["clk64_mhz"]),
                     "clock_corrected_basis": f"{sms} SMs x "
                                              f"{TENSOR_FLOP_PER_CLK_SM[w.dtype]:.0f} FLOP/clk "
                                              f"x clk64_mhz"},
        "clocks": {**t["clocks"], "clk64_mhz": t["clk64_mhz"], "clk64_ctas": t["ctas"],
                   "window": "nvidia-smi: soak + timed steps; clk64: the timed kernels' CTAs "
                             "(clock64 / %globaltimer)"},
        "hbm": hbm_figure(plan, ms_per_step, peaks),
        "gpu_launches": args.steps * plan.launches,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "step_ms_min": min(times_ms), "step_ms_median": statistics.median(times_ms),
        "other_workloads": other,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
