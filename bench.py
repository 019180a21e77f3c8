"""Benchmark: causal FP8 prefill attention TFLOP/s at S=32K, D=128 (and % of the GB300 FP8 peak).

One step = one zyfa_attn_fwd_causal call over the whole workload B=1, H=32, H_kv=8, S=32768, D=128
(Gaussian inputs quantised to e4m3 with per-tensor descales).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--dtype fp8|bf16] [--config bench32k|mla32k|...]
  python bench.py --impl reference ...     # the CPU oracle on the host cores, same metric and workload
  python bench.py --mma-rate               # the GPU's dense FP8 / BF16 tensor-core rate (the peak's measurement)

FLOP convention: ``value`` counts the algorithmic causal FLOPs B*H*S^2*(D_qk+D_v) (half the dense count,
what the tensor cores must execute); ``value_dense_formula`` reports the 2*B*H*S^2*(D_qk+D_v) variant.
Under torchrun (N > 1) every rank runs its own replica of the workload (no data exchange); ``value``
is the sum over ranks of the FLOPs divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal FP8 prefill attention TFLOP/s at S=32K D=128 and % of GB300 FP8 peak"
# Nominal dense tensor peaks (PFLOP/s) used only for the FP8:BF16 ratio applied to the measured bf16 peak.
NOMINAL_RATIO_FP8_TO_BF16 = 4.5 / 2.25
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# Dense tcgen05 MMA rate per SM and cycle of this GPU, as `bench.py --mma-rate` measures it (clock64
# spans of back-to-back M=128, N=256 products): the kernel's fraction of the tensor core's own rate at
# the clock sampled during the timed region.
MMA_FLOP_PER_CYCLE_PER_SM = {"fp8": 16384, "bf16": 8192}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["zyfa", "reference"], default="zyfa")
    ap.add_argument("--dtype", choices=["fp8", "bf16"], default="fp8")
    ap.add_argument("--config", default="bench32k")
    ap.add_argument("--heads", type=int, default=0, help="override H (profiling a smaller case)")
    ap.add_argument("--seq", type=int, default=0, help="override S (a sequence-length sweep)")
    ap.add_argument("--no-energy", action="store_true",
                    help="skip the energy record (NVML total-energy counter around a loop of >= --energy-seconds)")
    ap.add_argument("--energy-seconds", type=float, default=1.0)
    ap.add_argument("--hadamard", action="store_true",
                    help="also time the Hadamard rotation + quantisation pre-pass of Q and K (bf16 in)")
    ap.add_argument("--p-mode", choices=["lean", "exact", "exact-noblock"], default="lean",
                    help="FP8 probabilities: Lean P (the method), exact exponential (the ablation), or exact "
                         "without the per-block scaling")
    ap.add_argument("--mma-rate", action="store_true",
                    help="measure the dense FP8 and BF16 tcgen05 MMA rate (burst and sustained) instead")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--host-chunks", type=int, default=0,
                    help="chunks of the host-buffer call in the e2e leg (0 = the library's plan: six chunks, four "
                         "equal ones and two short tails, from 32 query blocks of 256 rows; else four)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle sample")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def library_host_chunks(S):
    """Chunks the host-buffer entry point uses for chunks = 0 (its documented plan): from 32 query
    blocks of 256 rows, four equal chunks and two short tails; below that, four equal chunks (at most
    one per block)."""
    nqb = (S + 255) // 256
    return 6 if nqb >= 32 else min(4, nqb)


def kernel_source_hash():
    """Hash of the kernel sources; recorded ncu traffic counts only while it matches."""
    import hashlib
    h = hashlib.sha256()
    for f in ("zyfa_fwd.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "fp8_causal_prefill_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def shape_for(args):
    from fp8_causal_prefill_gb300.inputs import CONFIGS, Shape
    sh = CONFIGS[args.config]
    if args.heads:
        hkv = max(1, args.heads * sh.H_kv // sh.H)
        sh = Shape(sh.B, sh.S, args.heads, hkv, sh.D_qk, sh.D_v, sh.kind)
    if args.seq:
        sh = Shape(sh.B, args.seq, sh.H, sh.H_kv, sh.D_qk, sh.D_v, sh.kind)
    return sh


def workload_name(sh, dtype, p_mode="lean"):
    extra = {"exact": ", exact-P ablation", "exact-noblock": ", exact-P ablation without block scaling"}.get(
        p_mode, "") if dtype == "fp8" else ""
    return (f"{'e4m3' if dtype == 'fp8' else 'bf16'} causal prefill B={sh.B} H={sh.H} H_kv={sh.H_kv} S={sh.S} "
            f"D_qk={sh.D_qk} D_v={sh.D_v} {sh.kind} inputs{extra}")


NVML_CLOCK_SM = 1
# clock event (throttle) reason bits of NVML's public API that bear on a measurement
NVML_REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}


def _device_uuid(dev_index):
    try:
        import torch
        if torch.cuda.is_available():
            u = getattr(torch.cuda.get_device_properties(dev_index), "uuid", None)
            return None if u is None else str(u)
    except Exception:  # noqa: BLE001 - no device, no uuid: fall back to the index
        pass
    return None


class Nvml:
    """Read-only NVML queries for one GPU through ctypes: SM clock, maximum SM clock, board power,
    clock event reasons and the cumulative board energy.  Nothing is set.  ``lib`` replaces
    libnvidia-ml (tests pass a fake); ``ok`` is False when NVML cannot be used."""

    def __init__(self, cuda_index, nvml_index=None, lib=None):
        import ctypes
        self.c = ctypes
        self.lib = None
        self.h = ctypes.c_void_p()
        try:
            lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            # the CUDA device's UUID names the same board in NVML; the index is the fallback
            uuid = _device_uuid(cuda_index)
            ok = uuid is not None and lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(),
                                                                      ctypes.byref(self.h)) == 0
            if not ok:
                idx = cuda_index if nvml_index is None else nvml_index
                ok = lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) == 0
            if ok:
                self.lib = lib
        except (OSError, AttributeError):
            self.lib = None

    @property
    def ok(self):
        return self.lib is not None

    def _query(self, fn_names, ctype, *args):
        if self.lib is None:
            return None
        for name in fn_names:
            fn = getattr(self.lib, name, None)
            if fn is None:
                continue
            v = ctype(0)
            return int(v.value) if fn(self.h, *args, self.c.byref(v)) == 0 else None
        return None

    def sm_mhz(self):
        return self._query(("nvmlDeviceGetClockInfo",), self.c.c_uint, NVML_CLOCK_SM)

    def sm_max_mhz(self):
        return self._query(("nvmlDeviceGetMaxClockInfo",), self.c.c_uint, NVML_CLOCK_SM)

    def power_w(self):
        mw = self._query(("nvmlDeviceGetPowerUsage",), self.c.c_uint)
        return None if mw is None else mw / 1000.0

    def reasons_mask(self):
        return self._query(("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"),
                           self.c.c_ulonglong)

    def energy_mj(self):
        return self._query(("nvmlDeviceGetTotalEnergyConsumption",), self.c.c_ulonglong)


class EnergyCounter:
    """Cumulative board energy of one GPU from NVML (read only), millijoules."""

    def __init__(self, cuda_index, nvml_index=None, lib=None):
        self.nvml = Nvml(cuda_index, nvml_index, lib)

    def read_mj(self):
        return self.nvml.energy_mj()


def energy_block(e_start_mj, e_end_mj, steps, flops_per_step, seconds):
    """Energy per step and TFLOP per joule from two readings of the cumulative energy counter around
    `steps` steps that took `seconds`; an `unavailable` record when the counter gave nothing usable."""
    if e_start_mj is None or e_end_mj is None or e_end_mj <= e_start_mj or steps <= 0 or seconds <= 0:
        return {"unavailable": "NVML energy counter not readable on this box"}
    joules = (e_end_mj - e_start_mj) * 1e-3
    return {"joules_per_step": joules / steps, "tflop_per_joule": flops_per_step * steps / joules / 1e12,
            "avg_power_w": joules / seconds, "steps": steps, "seconds": seconds,
            "method": "NVML total-energy counter (board), read before and after the loop"}


def summarize_clocks(rows, window, source):
    """Clock record of a timed region from samples (wall time, SM MHz, max SM MHz, power W or None,
    set of active reason names): only samples inside the window count, unless there are none."""
    inside = [r for r in rows if window and window[0] <= r[0] <= window[1]]
    used = inside if inside else rows
    reasons = set().union(*[r[4] for r in used]) if used else set()
    sm = [r[1] for r in used]
    power = [r[3] for r in used if r[3] is not None]
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_mhz_min": min(sm) if sm else None,
            "sm_max_mhz": max(r[2] for r in used) if used else None,
            "power_w_median": statistics.median(power) if power else None, "samples": len(sm),
            "samples_in_window": bool(inside), "reasons": sorted(reasons), "source": source}


class NvmlSampler:
    """SM clock, power and clock event reasons from NVML every `period` seconds on a host thread
    (read-only queries); only samples stamped inside the timed region are summarised."""

    def __init__(self, nvml, period=0.005):
        self.nvml = nvml
        self.period = period
        self.rows = []
        self.window = None
        self._stop = None
        self._thread = None

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def sample(self):
        sm = self.nvml.sm_mhz()
        if sm is None:
            return
        mask = self.nvml.reasons_mask() or 0
        names = {n for n, bit in NVML_REASONS.items() if mask & bit}
        self.rows.append((time.time(), float(sm), float(self.nvml.sm_max_mhz() or 0), self.nvml.power_w(), names))

    def start(self):
        import threading
        self._stop = threading.Event()

        def run():
            while not self._stop.is_set():
                self.sample()
                self._stop.wait(self.period)
        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()
        time.sleep(0.05)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        return summarize_clocks(self.rows, self.window, f"NVML every {self.period * 1e3:g} ms")


class ClockSampler:
    """nvidia-smi sampled every 50 ms (used when NVML cannot be loaded in-process); only samples stamped
    inside the timed region (host wall clock, from the launch of the first timed step to the
    synchronize after the last) are summarised."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.window = None

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="zyfa_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                vals = (float(parts[1]), float(parts[2]))
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = None
            rows.append((ts, vals[0], vals[1], pw, parts[5:9]))
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = [(r[0], r[1], r[2], r[3], {n for n, v in zip(names, r[4]) if v.lower().startswith("active")})
                for r in rows]
        return summarize_clocks(rows, self.window, "nvidia-smi every 50 ms")


def slowest_rank_ms(local_ms: float, world: int, device) -> float:
    """The step time of the job: the maximum over ranks of each rank's own CUDA-event time."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica, so the work adds up over ranks and the
    slowest rank's time is the job's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def cpu_oracle_sample(p, dtype, budget_s):
    """Time the oracle on a seeded sample of query rows of the workload (rows are independent)."""
    import numpy as np

    import oracle as O

    sh = p.shape
    sc = O.default_softmax_scale(sh.D_qk)
    rng = np.random.default_rng(123)
    done_rows, flops, elapsed, calls = 0, 0.0, 0.0, 0
    while elapsed < budget_s and calls < 64:
        rows = np.sort(rng.choice(sh.S, size=min(sh.S, 256), replace=False))
        head = int(rng.integers(0, sh.H))
        t0 = time.perf_counter()
        if dtype == "fp8":
            O.leanp_causal_attention(p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, sc, rows=rows,
                                     heads=[head])
        else:
            f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
            O.bf16_causal_attention(f(p.qb), f(p.kb), f(p.vb), sc, rows=rows, heads=[head])
        elapsed += time.perf_counter() - t0
        flops += float(np.sum(2.0 * (rows + 1) * (sh.D_qk + sh.D_v))) * sh.B
        done_rows += len(rows)
        calls += 1
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done_rows} query rows x 1 head of {workload_name(sh, dtype)} "
                      f"(seeded uniform rows, {flops:.3e} causal FLOPs in {elapsed:.1f} s; numpy float64, "
                      f"BLAS threads = cores)"}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded row sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from fp8_causal_prefill_gb300.inputs import make_problem

    sh = shape_for(args)
    p = make_problem(sh, seed=0, bf16=(args.dtype == "bf16"), fp8=(args.dtype == "fp8"))
    per_step = max(0.5, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(p, args.dtype, per_step / 4)
    vals = [cpu_oracle_sample(p, args.dtype, per_step) for _ in range(args.steps)]
    value = statistics.median(v["value"] for v in vals)
    cpu = dict(vals[-1])
    cpu["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(sh, args.dtype), "sample": cpu["sample"]},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def make_sampler(cuda_index, nvml_index):
    """The clock record's sampler: NVML in-process every 5 ms, else nvidia-smi every 50 ms."""
    nv = Nvml(cuda_index, nvml_index)
    return NvmlSampler(nv) if nv.ok else ClockSampler(nvml_index)


def run_mma_rate(args):
    """Dense tensor-core rate of this GPU with the attention kernel's MMA forms: one CTA per SM issuing
    M=128, N=256 MMAs from shared memory (zyfa_probe_mma_rate).  A burst of ten launches and a loop of
    at least three seconds (where the board's power cap sets the clock); CUDA events for the rate,
    each CTA's clock64 span for FLOP per cycle per SM."""
    import torch

    from fp8_causal_prefill_gb300 import api

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = api.load_library()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    smi_index = 0
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    if visible and visible[0].strip().isdigit():
        smi_index = int(visible[0])
    line = {"probe": "dense tcgen05 MMA rate, M=128 N=256, operands in shared memory, one CTA per SM",
            "sms": nsm}
    for name, fp8, iters in (("fp8_e4m3", 1, 20000), ("bf16", 0, 10000)):
        fpi = lib.zyfa_probe_mma_flops_per_iter(fp8)
        cycles = torch.zeros(nsm, dtype=torch.int64, device=dev)
        flag = torch.zeros(1, dtype=torch.int32, device=dev)

        def launch():
            st = lib.zyfa_probe_mma_rate(fp8, iters, nsm, cycles.data_ptr(), flag.data_ptr(), sptr)
            if st != 0:
                raise api.ZyfaError(st, "zyfa_probe_mma_rate")
        for _ in range(3):
            launch()
        torch.cuda.synchronize(dev)
        res = {}
        for mode, n in (("burst", 10), ("sustained", None)):
            sampler = make_sampler(0, smi_index)
            sampler.start()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if n is None:   # enough launches for about three seconds at the burst rate
                n = max(10, int(3.0 / (res["burst_ms_per_launch"] * 1e-3)))
            t0 = time.time()
            e0.record(stream)
            for _ in range(n):
                launch()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            sampler.mark(t0, time.time())
            clk = sampler.stop()
            ms = e0.elapsed_time(e1) / n
            cyc = int(cycles.max().item())
            res[f"{mode}_ms_per_launch"] = ms
            res[f"{mode}_tflops"] = fpi * iters * nsm / (ms * 1e-3) / 1e12
            res[f"{mode}_launches"] = n
            res[f"{mode}_sm_mhz"] = clk.get("sm_mhz")
            res[f"{mode}_clock_reasons"] = clk.get("reasons")
            res[f"{mode}_flop_per_cycle_per_sm"] = fpi * iters / cyc
        if int(flag.item()) != 0:
            res["timed_out"] = True
        fpc = res["burst_flop_per_cycle_per_sm"]
        res["tflops_at_2070_mhz"] = fpc * nsm * 2070e6 / 1e12
        line[name] = res
    # the attention kernel's own MMA forms, each alone (zyfa_probe_mma_form_rate): FLOP per cycle per SM
    # from the CTAs' clock64 spans, as a fraction of the dense rate of its type measured above
    forms = {}
    names = ("fp8_score_ss_n128", "fp8_pv_block_scaled_ts_n144", "fp8_score_then_pv", "fp8_score_two_n64_halves",
             "bf16_score_ss_n128", "bf16_score_ss_n64_d192")
    for form, fname in enumerate(names):
        fpi = lib.zyfa_probe_mma_form_flops_per_iter(form)
        iters = 5000
        cycles = torch.zeros(nsm, dtype=torch.int64, device=dev)
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(3):
            st = lib.zyfa_probe_mma_form_rate(form, iters, nsm, cycles.data_ptr(), flag.data_ptr(), sptr)
            if st != 0:
                raise api.ZyfaError(st, "zyfa_probe_mma_form_rate")
        torch.cuda.synchronize(dev)
        fpc = fpi * iters / int(cycles.max().item())
        dense = line["bf16" if fname.startswith("bf16") else "fp8_e4m3"]["burst_flop_per_cycle_per_sm"]
        forms[fname] = {"flop_per_cycle_per_sm": fpc, "frac_of_dense": fpc / dense,
                        "timed_out": int(flag.item()) != 0}
    line["kernel_mma_forms"] = forms
    print(json.dumps(line), flush=True)
    return 0


def main():
    import numpy as np

    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.mma_rate:
        return run_mma_rate(args)

    import torch
    import torch.distributed as dist

    from fp8_causal_prefill_gb300 import api
    from fp8_causal_prefill_gb300.inputs import make_problem

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    sh = shape_for(args)
    p = make_problem(sh, seed=rank, bf16=(args.dtype == "bf16"), fp8=(args.dtype == "fp8"))
    if args.dtype == "fp8":
        host = [t.contiguous() for t in (p.q8, p.k8, p.v8)]
        dtype_code = api.ZYFA_DTYPE_E4M3
    else:
        host = [t.contiguous() for t in (p.qb, p.kb, p.vb)]
        dtype_code = api.ZYFA_DTYPE_BF16
    dq, dk, dv = (t.to(dev) for t in host)
    desc = torch.tensor([p.dq, p.dk, p.dv], dtype=torch.float32, device=dev)
    out = torch.empty((sh.B, sh.S, sh.H, sh.D_v), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    api.load_library()

    p_mode = {"exact": api.ZYFA_P_EXACT, "exact-noblock": api.ZYFA_P_EXACT_NO_BLOCK_SCALE}.get(args.p_mode,
                                                                                              api.ZYFA_P_LEAN)

    def step(q, k, v, o):
        st = api.zyfa_attn_fwd_causal_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), sh.B, sh.S, sh.H,
                                         sh.H_kv, sh.D_qk, sh.D_v, 0.0, dtype_code,
                                         desc.data_ptr() if args.dtype == "fp8" else 0,
                                         desc.data_ptr() + 4 if args.dtype == "fp8" else 0,
                                         desc.data_ptr() + 8 if args.dtype == "fp8" else 0, p_mode=p_mode,
                                         stream=sptr)
        if st != 0:
            raise api.ZyfaError(st, "zyfa_attn_fwd_causal_ex")

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    flops = sh.causal_flops                      # per step per rank
    for _ in range(max(3, args.warmup)):
        step(dq, dk, dv, out)
    barrier()

    smi_index = local
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    if local < len(visible) and visible[local].strip().isdigit():
        smi_index = int(visible[local])
    sampler = make_sampler(local, smi_index) if rank == 0 else None
    if rank == 0:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    # L2 (129 MB): a working set that fits is flushed between timed steps by writing 256 MB, and the
    # steps are then timed one by one (the flush is outside every step's events)
    work_bytes = sum(t.numel() * t.element_size() for t in (dq, dk, dv, out))
    flush = work_bytes < (256 << 20)
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    barrier()
    t_wall0 = time.time()
    for i in range(args.steps):
        if flush:
            scrub.fill_(i & 0xFF)
        starts[i].record(stream)
        step(dq, dk, dv, out)
        ends[i].record(stream)
    barrier()
    clocks = None
    if rank == 0:
        sampler.mark(t_wall0, time.time())
        clocks = sampler.stop()
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(kernel_ms) if flush else starts[0].elapsed_time(ends[-1])
    ms_per_step = slowest_rank_ms(total_ms, world, dev) / args.steps
    value = job_throughput(flops, world, ms_per_step)
    zst = api.zyfa_check_errors(sptr)
    if zst != 0:
        raise api.ZyfaError(zst, "kernel status")

    # energy per step: NVML's cumulative energy counter (read only) around a loop of at least
    # --energy-seconds (the counter moves in steps too coarse for a window of a few milliseconds)
    energy = None
    if not args.no_energy and rank == 0:
        meter = EnergyCounter(local, smi_index)
        n_en = max(args.steps, int(args.energy_seconds / max(ms_per_step * 1e-3, 1e-6)) + 1)
        e_start = meter.read_mj()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(n_en):
            step(dq, dk, dv, out)
        g1.record(stream)
        torch.cuda.synchronize(dev)
        energy = energy_block(e_start, meter.read_mj(), n_en, flops, g0.elapsed_time(g1) * 1e-3)

    # the Hadamard pre-pass of Q and K (bf16 -> rotated e4m3 + descale), timed on its own
    prepass = None
    if args.hadamard:
        from fp8_causal_prefill_gb300.inputs import make_problem as _mk
        pb = p if p.qb is not None else _mk(sh, seed=rank, bf16=True, fp8=False)
        xq, xk = pb.qb.to(dev), pb.kb.to(dev)
        qr, kr = xq.numel() // sh.D_qk, xk.numel() // sh.D_qk
        c8 = [torch.empty(x.shape, dtype=torch.uint8, device=dev) for x in (xq, xk)]
        dsc = torch.empty(2, dtype=torch.float32, device=dev)
        wsb = api.zyfa_hadamard_workspace_bytes(qr) + api.zyfa_hadamard_workspace_bytes(kr)
        ws = torch.empty(max(1, wsb // 4), dtype=torch.float32, device=dev)

        def prestep():
            # Q and K in one launch per pass
            st = api.zyfa_hadamard_quantize_qk_e4m3(xq.data_ptr(), c8[0].data_ptr(), dsc.data_ptr(), qr,
                                                    xk.data_ptr(), c8[1].data_ptr(), dsc.data_ptr() + 4, kr,
                                                    sh.D_qk, ws.data_ptr(), ws.numel() * 4, sptr)
            if st != 0:
                raise api.ZyfaError(st, "zyfa_hadamard_quantize_qk_e4m3")
        for _ in range(3):
            prestep()
        barrier()
        n_pre = 20
        # back to back (the inputs, 335 MB at 32K, exceed L2; launches overlap at step boundaries)
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(n_pre):
            prestep()
        h1.record(stream)
        # each step timed on its own after a 256 MB write (outside its events): no step starts on
        # rows the previous one left in L2, and no launch overlaps the previous step
        pre_scrub = scrub if scrub is not None else torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        hs = [torch.cuda.Event(enable_timing=True) for _ in range(n_pre)]
        he = [torch.cuda.Event(enable_timing=True) for _ in range(n_pre)]
        for i in range(n_pre):
            pre_scrub.fill_(i & 0xFF)
            hs[i].record(stream)
            prestep()
            he[i].record(stream)
        barrier()
        pre_b2b_ms = h0.elapsed_time(h1) / n_pre
        pre_ms = sum(a.elapsed_time(b) for a, b in zip(hs, he)) / n_pre
        del pre_scrub
        elems = xq.numel() + xk.numel()
        alg_bytes = 3 * elems      # bf16 read once + e4m3 written once
        moved = 5 * elems          # two passes read the bf16 input
        hbm = load_peaks()[0].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        prepass = {"ms": pre_ms, "ms_back_to_back": pre_b2b_ms, "fraction_of_attention": pre_ms / ms_per_step,
                   "algorithmic_bytes": alg_bytes, "bytes_moved": moved,
                   "achieved_gbs": moved / (pre_ms * 1e-3) / 1e9,
                   "hbm_frac": moved / (pre_ms * 1e-3) / 1e9 / hbm,
                   "launches_per_step": 2,
                   "l2": "ms: flushed before every step (256 MB write outside the events); ms_back_to_back: 20 steps in a row",
                   "what": "Q and K of the workload, bf16 -> rotated e4m3 + descale"}

    # end to end through the same C entry point with host buffers: H2D of q/k/v, the call, D2H of out
    e2e = None
    if not args.no_e2e:
        hpin = [h.pin_memory() for h in host]
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(h.numel() * h.element_size() for h in hpin) + (12 if args.dtype == "fp8" else 0)
        hdesc = torch.tensor([p.dq, p.dk, p.dv], dtype=torch.float32).pin_memory()
        d2h = hout.numel() * hout.element_size()
        n_e2e = max(3, min(args.steps, 20))
        dptr = desc.data_ptr() if args.dtype == "fp8" else 0

        def host_step():
            # the public host-buffer call: uploads of q/k/v, chunked kernels and the download of out,
            # overlapped on the library's copy streams; the descales are uploaded first
            if args.dtype == "fp8":
                desc.copy_(hdesc, non_blocking=True)
            st = api.zyfa_attn_fwd_causal_host(hpin[0].data_ptr(), hpin[1].data_ptr(), hpin[2].data_ptr(),
                                               hout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                               out.data_ptr(), sh.B, sh.S, sh.H, sh.H_kv, sh.D_qk, sh.D_v, 0.0,
                                               dtype_code, dptr, dptr + 4 if dptr else 0, dptr + 8 if dptr else 0,
                                               args.host_chunks, sptr)
            if st != 0:
                raise api.ZyfaError(st, "zyfa_attn_fwd_causal_host")
        for _ in range(3):
            host_step()
        barrier()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
        ev[0].record(stream)
        for i in range(n_e2e):
            host_step()
            ev[i + 1].record(stream)
        barrier()
        step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(n_e2e)]
        te = slowest_rank_ms(ev[0].elapsed_time(ev[-1]) / n_e2e, world, dev)
        e2e = {"value": job_throughput(flops, world, te), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": te,
               "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
               "steps": n_e2e, "call": "zyfa_attn_fwd_causal_host (pinned host buffers)",
               "chunks": args.host_chunks or library_host_chunks(sh.S),
               "plan": "given" if args.host_chunks else "library default"}

    far_fraction = None
    if rank == 0 and sh.kind == "mistral" and p.q is not None:
        # the outlier recipe stands in for captured activations: report how many (row, 64-key block)
        # pairs sit more than 8 binades below the row maximum (a seeded sample of rows, head 0)
        import numpy as _np

        from fp8_causal_prefill_gb300.inputs import far_block_fraction
        rows = _np.sort(_np.random.default_rng(5).choice(sh.S, size=min(sh.S, 64), replace=False))
        far_fraction = far_block_fraction(p, rows)
    if rank == 0:
        peaks, src = load_peaks()
        is_fp8 = args.dtype == "fp8"
        ratio = NOMINAL_RATIO_FP8_TO_BF16 if is_fp8 else 1.0
        peak = peaks["bf16_tflops"] * ratio
        peak_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio
        avg_kernel_ms = statistics.fmean(kernel_ms)
        achieved = flops / (avg_kernel_ms * 1e-3) / 1e12
        traffic = None
        tpath = os.path.join(ROOT, "profiles", "dram_traffic.json")
        if os.path.exists(tpath):
            with open(tpath) as f:
                td = json.load(f)
            key = f"{args.dtype}:{args.config}" + (f":{args.p_mode}" if args.p_mode != "lean" else "")
            if key in td and not args.heads and not args.seq and td[key].get("kernel_sha256") == kernel_source_hash():
                traffic = td[key].get("bytes_per_launch")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if is_fp8 else "bf16", "data": "synthetic",
            "config": {"workload": workload_name(sh, args.dtype, args.p_mode),
                       "l2": (f"working set {work_bytes / 1e6:.0f} MB is under twice the 129 MB L2: flushed between "
                              f"steps (256 MB write outside the timed events; value from per-step events)" if flush else
                              f"working set {work_bytes / 1e6:.0f} MB (inputs + output) exceeds the 129 MB L2; "
                              f"no flush"),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       **({"far_block_fraction": far_fraction} if far_fraction is not None else {})},
            "value_dense_formula": 2.0 * value,
            "pct_of_fp8_peak": 100.0 * value / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": (f"{src}: bf16 burst {peaks['bf16_tflops']} TFLOP/s x {ratio:g} "
                                         f"(nominal {'fp8' if is_fp8 else 'bf16'}/bf16 ratio)"),
                         "frac_of_sustained": achieved / peak_sus},
            "kernel_ms": {"mean": avg_kernel_ms, "median": statistics.median(kernel_ms),
                          "p10": float(np.percentile(kernel_ms, 10)), "p90": float(np.percentile(kernel_ms, 90)),
                          "min": min(kernel_ms), "max": max(kernel_ms)},
            "gpu_launches": args.steps * api.zyfa_kernel_launches(sh.B, sh.S, sh.H),
            "clocks": clocks,
        }
        if clocks is not None and clocks.get("sm_mhz"):
            # step time x median SM clock: the step in thousands of SM cycles, comparable across clocks
            clocks["kcycles_per_step"] = ms_per_step * clocks["sm_mhz"]
            nsm = torch.cuda.get_device_properties(dev).multi_processor_count
            hw = MMA_FLOP_PER_CYCLE_PER_SM[args.dtype] * nsm * clocks["sm_mhz"] * 1e6 / 1e12
            line["roofline"]["tensor_rate_at_clock"] = hw
            line["roofline"]["frac_of_tensor_rate"] = achieved / hw
        if e2e is not None:
            line["e2e"] = e2e
        if prepass is not None:
            line["hadamard_prepass"] = prepass
        if energy is not None:
            line["energy"] = energy
        if not args.no_cpu and world == 1:
            line["cpu_baseline"] = cpu_oracle_sample(p, args.dtype, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
