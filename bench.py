#!/usr/bin/env python3
"""Throughput of the GDN speculative-verify hot path on one GB300 (or N independent replicas).

Workload (the metric's configuration): one GDN layer with Hk=16, Hv=32, dk=dv=128, a width-4
conv over 8192 packed bf16 channels, fp32 state; 64 speculative rows of 4 verify tokens
(3 drafts), num_accepted uniform in [1, 4], distinct slots in a 512-slot pool with 5% of the
spec_state_indices entries NULL.  A step is one pass of the whole path over that batch:
gdn_mixed_batch (conv update, then the gated delta rule with per-token state stores).

Output: one JSON line (rank 0).  `value` = verify tokens processed per second over the timed
steps (device time, CUDA events on the launching stream, L2 flushed between steps); `e2e` =
the same metric through gdn_mixed_batch with the step's inputs copied from pinned host memory
and its outputs copied back inside the timed region; `roofline` = the recurrence kernel's
algorithmic bytes per launch / its event-timed duration against the measured HBM copy
bandwidth; `cpu_baseline` = the CPU oracle timed on this host's cores on the same workload.
``--impl reference`` times the CPU oracle alone (the reference arm of this comparison).
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

import torch  # noqa: E402

METRIC = "GDN spec-verify tokens/s per layer; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
WORKLOAD = ("spec_verify: 1 GDN layer Hk=16 Hv=32 dk=dv=128, conv width 4 over 8192 bf16 channels, fp32 state; "
            "64 rows x 4 verify tokens (3 drafts), num_accepted U[1,4], 512-slot pool, 5% NULL slots")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")

# Other workloads (parity configurations) can be timed for profiling; the metric's line is spec_verify.
WORKLOADS = {
    "spec_verify": WORKLOAD,
    "non_spec_decode": "non_spec_decode: same layer, 64 one-token non-spec rows, 256-slot pool",
    "mixed": "mixed: same layer, 8 decode rows first, 32 spec rows of 4 tokens and prefill rows of 512 and 1024 "
             "tokens interleaved",
    "long_prefill": "long_prefill: same layer, one 8192-token prefill row continuing a prior state",
}


# Seeded index sets the timed steps rotate over (slots, acceptance counts, NULL positions and
# activations differ; the distributions are the workload's).  The first is the parity workload.
INDEX_SETS = {"spec_verify": (2, 1002, 2002, 3002), "non_spec_decode": (1, 1001, 2001, 3001),
              "mixed": (3, 1003, 2003, 3003), "long_prefill": (20,)}


def make_workload(name, seed=None):
    from gated_deltanet_linear_spec_gb300 import workloads
    seed = INDEX_SETS[name][0] if seed is None else seed
    return {"spec_verify": workloads.spec_verify, "non_spec_decode": workloads.non_spec_decode,
            "mixed": workloads.mixed, "long_prefill": lambda seed: workloads.long_prefill(8192, seed)}[name](seed=seed)


def workload_config(args) -> dict:
    """The workload a line is quoted on: identical keys and values in both arms."""
    return {"workload": WORKLOADS[args.workload], "index_sets": len(INDEX_SETS[args.workload]),
            "qkv_layout": args.qkv_layout, "conv_layout": args.conv_layout}


def source_hash(*names) -> str:
    """Hash of the kernel sources with comments and blank space removed, so that traffic recorded
    for a kernel stays attached to it until its code changes."""
    import hashlib
    import re
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_deltanet_linear_spec_gb300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                    and parts[2] == src_hash:
                return int(parts[3])
    return None


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


# ------------------------------------------------------------------------------------------
# algorithmic bytes (from the actual index tensors)

def algorithmic_bytes(batch) -> dict:
    L = batch.layer
    C, Hv, dv, dk, W = L.channels, L.num_v_heads, L.head_v_dim, L.head_k_dim, L.conv_width
    act = 2 if L.act_dtype == torch.bfloat16 else 4
    state = Hv * dv * dk * 4
    loads = stores = conv = 0
    for sub in (batch.spec, batch.non_spec):
        if sub is None:
            continue
        qsl = sub.query_start_loc.tolist()
        for n in range(sub.num_seqs):
            ln = qsl[n + 1] - qsl[n]
            if ln == 0:
                continue
            if sub.is_spec:
                ssi = sub.spec_state_indices[n].tolist()
                na = int(sub.num_accepted_tokens[n])
                loads += ssi[na - 1] > 0
                stores += sum(1 for t in range(ln) if ssi[t] > 0)
                if L.conv_layout == 1:  # one W-1 snapshot read, one written per non-NULL verify slot
                    conv += ((W - 1) * (ssi[na - 1] > 0) + (W - 1) * sum(ssi[t] > 0 for t in range(ln))) * C * act
                elif ssi[0] > 0:
                    conv += (W - 1 + W - 2 + ln) * C * act
            else:
                s = int(sub.state_indices[n])
                hi = 1 if sub.has_initial_state is None else int(sub.has_initial_state[n])
                src = s
                if sub.num_accepted_tokens is not None:  # acceptance-aware rows load the accepted state
                    src = int(sub.spec_state_indices[n, int(sub.num_accepted_tokens[n]) - 1])
                loads += (src > 0 and hi != 0)
                stores += s > 0
                conv_src = src if (sub.num_accepted_tokens is not None and L.conv_layout == 1) else s
                conv += ((W - 1) * (conv_src > 0 and hi != 0) + (W - 1) * (s > 0)) * C * act
    T = batch.num_actual_tokens
    ssm = (loads + stores) * state
    io = T * (C * act + 2 * Hv * act + Hv * dv * act)
    params = C * W * act + 2 * Hv * 4
    rec = ssm + T * (2 * Hv * act + Hv * dv * act)  # what the recurrence kernel must move
    return {"total": ssm + io + conv + params, "ssm": ssm, "recurrence": rec, "conv": conv,
            "state_loads": loads, "state_stores": stores}


# ------------------------------------------------------------------------------------------
# clocks during the timed region

# The sampling loop, run as a child process so that no lock of this interpreter delays it: read-only
# NVML queries of one GPU (SM clock, its maximum, the clock-event reasons) every `period` seconds
# on the system-wide monotonic clock, written out when the stop file appears.
_NVML_SAMPLER = r"""
import ctypes, os, sys, time
uuid, index, period, out_path, stop_path = sys.argv[1], int(sys.argv[2]), float(sys.argv[3]), sys.argv[4], sys.argv[5]
lib = ctypes.CDLL("libnvidia-ml.so.1")
if lib.nvmlInit_v2() != 0:
    sys.exit(3)
h = ctypes.c_void_p()
if not uuid or lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
    if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
        sys.exit(4)
reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # the maximum does not change
    sys.exit(5)
rows = []
print("ready", flush=True)
while not os.path.exists(stop_path) and len(rows) < 2000000:
    t = time.monotonic()
    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and reasons(h, ctypes.byref(rs)) == 0:
        rows.append("%.6f %d %d %d" % (t, sm.value, mx.value, rs.value))
    time.sleep(period)
with open(out_path, "w") as f:
    f.write("\n".join(rows))
lib.nvmlShutdown()
"""


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons sampled during the run by read-only NVML
    queries in a child process, as fast as NVML answers (at most every 0.25 ms; on GB300 hosts
    with the GPU busy about every 5-10 ms, so a timed region of a few milliseconds holds one or
    two samples and the whole run's samples are reported beside them).  A sampling thread in this interpreter
    competed with the launching thread for the interpreter lock (1 us more per spec-verify
    step); the child does not.  nvidia-smi's 200 ms polling when NVML cannot be loaded.  Times
    are on the system-wide monotonic clock.  Nothing here changes a setting of the GPU."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int, period_s: float = 0.00025):
        self.samples = []  # (monotonic time, sm_mhz, max_mhz, reason names)
        self.windows = []  # (start, end) of the metric's timed region
        self.source = None
        self.period_ms = period_s * 1e3
        self._child = None
        self._smi = None
        if not self._start_nvml(cuda_index, period_s):
            self._start_smi(cuda_index)

    def _start_nvml(self, cuda_index, period_s) -> bool:
        uuid = ""
        try:
            u = str(torch.cuda.get_device_properties(cuda_index).uuid)
            uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        try:
            self._dir = tempfile.mkdtemp(prefix="clocks")
            self._out = os.path.join(self._dir, "samples.txt")
            self._stopfile = os.path.join(self._dir, "stop")
            self._child = subprocess.Popen([sys.executable, "-c", _NVML_SAMPLER, uuid, str(cuda_index), str(period_s),
                                            self._out, self._stopfile], stdout=subprocess.PIPE,
                                           stderr=subprocess.DEVNULL, text=True)
            if self._child.stdout.readline().strip() != "ready":
                self._child.wait(timeout=10)
                self._child = None
                return False
            self.source = "nvml"
            return True
        except Exception:
            self._child = None
            return False

    def _start_smi(self, cuda_index):
        try:
            fd, self._path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            self._fh = os.fdopen(fd, "w")
            self._smi = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(cuda_index), "-lms", "200"], stdout=self._fh,
                                         stderr=subprocess.DEVNULL)
            self._t0 = time.monotonic()
            self.source = "nvidia-smi"
        except Exception:
            self._smi = None

    def mark(self, start: float, end: float) -> None:
        """Records one timed region (time.monotonic() taken after the synchronizes around it)."""
        self.windows.append((start, end))

    def stop(self) -> dict:
        if self._child is not None:
            open(self._stopfile, "w").close()
            try:
                self._child.wait(timeout=20)
                with open(self._out) as f:
                    for line in f:
                        parts = line.split()
                        if len(parts) != 4:
                            continue
                        bits = int(parts[3])
                        names = tuple(n for bit, n in self.REASONS.items() if bits & bit)
                        self.samples.append((float(parts[0]), float(parts[1]), float(parts[2]), names))
            except Exception:
                self._child.kill()
        elif self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except Exception:
                self._smi.kill()
            self._fh.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            with open(self._path) as f:
                for i, line in enumerate(f):
                    parts = [q.strip() for q in line.split(",")]
                    try:
                        sm, mx = float(parts[1]), float(parts[2])
                    except (ValueError, IndexError):
                        continue
                    rs = tuple(n for n, v in zip(names, parts[5:9]) if v.lower() == "active")
                    self.samples.append((self._t0 + 0.2 * i, sm, mx, rs))
            os.unlink(self._path)
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        inside = [s for s in self.samples if any(a <= s[0] <= b for a, b in self.windows)]
        use = inside if inside else self.samples
        reasons = sorted({r for s in use for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in use) if use else None,
                "sm_max_mhz": max(s[2] for s in use) if use else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "samples_whole_run": len(self.samples),
                "sm_mhz_whole_run": statistics.median(s[1] for s in self.samples) if self.samples else None,
                "reasons_whole_run": sorted({r for s in self.samples for r in s[3]}),
                "source": self.source, "period_ms": self.period_ms if self.source == "nvml" else 200.0}


# ------------------------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)

def oracle_tokens_per_s(batch, budget_s: float = 12.0, heads=None) -> dict:
    """The CPU oracle as it stands, timed on this host's cores over a bounded sample: the whole
    workload (or a few v-heads of it, scaled to all heads), run repeatedly until budget_s has
    passed (at least 3 runs); the rate is taken from the median run."""
    from tests.oracle_run import np_act, run_oracle
    cores = len(os.sched_getaffinity(0))
    conv_pool, ssm_pool = np_act(batch.conv_pool), np_act(batch.ssm_pool)  # copied once, outside the timing
    Hv = batch.layer.num_v_heads
    frac = 1.0 if heads is None else (heads[1] - heads[0]) / Hv
    runs = []
    while (sum(runs) < budget_s or len(runs) < 3) and len(runs) < 2000:
        t0 = time.perf_counter()
        run_oracle(batch, heads=heads, nthreads=cores, conv_pool=conv_pool, ssm_pool=ssm_pool)
        runs.append(time.perf_counter() - t0)
    what = "all 32 v-heads" if heads is None else f"v-heads {heads[0]}..{heads[1] - 1} of {Hv}, scaled to all"
    # one single-thread pass of the same sample, for the per-core rate
    t0 = time.perf_counter()
    run_oracle(batch, heads=heads, nthreads=1, conv_pool=conv_pool, ssm_pool=ssm_pool)
    one = time.perf_counter() - t0
    tokens = batch.num_actual_tokens * frac
    return {"value": tokens / statistics.median(runs), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the full token set ({batch.num_actual_tokens} tokens), {what}, run {len(runs)}x "
                      f"({sum(runs):.1f} s on {cores} threads); rate of the median run",
            "mean_value": tokens * len(runs) / sum(runs),
            "single_thread_value": tokens / one, "cpu_model": cpu_model()}


def cpu_model() -> str:
    """The host CPU's model name, as the kernel reports it (empty when it does not)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip().lower() in ("model name", "cpu model"):
                    return v.strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip().lower() == "model name":
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return ""


# ------------------------------------------------------------------------------------------
# replicas: every rank runs the same workload on its own GPU; the job's time is the slowest rank

def reduce_max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank floats (identity without a process group)."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch in the slowest rank's time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


# ------------------------------------------------------------------------------------------

def prefill_flops(batch) -> float:
    """Algorithmic FLOPs of the chunked form over the prefill rows: per (64-token chunk, v-head)
    5 c^2 d + 3 c d^2 + c^3 / 6 multiply-adds (c = 64, d = 128), two FLOPs each."""
    c, d = 64, batch.layer.head_k_dim
    chunks = 0
    sub = batch.non_spec
    qsl = sub.query_start_loc.tolist()
    for n in range(batch.num_decodes, sub.num_seqs):
        chunks += -(-(qsl[n + 1] - qsl[n]) // c)
    return 2.0 * chunks * batch.layer.num_v_heads * (5 * c * c * d + 3 * c * d * d + c ** 3 / 6)


def timed(fn, steps, flush, stream):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def timed_rotating(fns, steps, flush, stream):
    """Per-step milliseconds (CUDA events on the launching stream); step i runs fns[i % len(fns)],
    and the L2 flush runs between steps, outside the events."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (a, b) in enumerate(ev):
        a.record(stream)
        fns[i % len(fns)]()
        b.record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def per_launch_rate(units_per_set, ms):
    """Median over the timed launches of each launch's rate (launch i processed
    units_per_set[i % n] units in ms[i] milliseconds), in units per second."""
    n = len(units_per_set)
    return statistics.median(units_per_set[i % n] / (ms[i] * 1e-3) for i in range(len(ms)))


def end_to_end(db, batch, stream, flush, steps, dist):
    """The metric through gdn_mixed_batch with the step's inputs copied from pinned host memory
    and its outputs copied back, the way a serving loop runs it: two device buffer sets share the
    pools; step i+1's host->device copies and step i-1's device->host read overlap step i's
    kernels (copies on their own streams, ordered by events; the kernels stay in order on the
    compute stream, which carries the state from step to step).  Also the serial sequence
    (copy in, compute, copy out) and the kernels alone back to back without the L2 flush."""
    from gated_deltanet_linear_spec_gb300.device_batch import to_device
    host_in = {k: getattr(db, k).cpu().pin_memory() for k in ("x", "a", "b")}
    idx = []
    for sub in (db.spec, db.non_spec):
        if sub is None:
            continue
        for k in ("query_start_loc", "token_indx", "state_indices", "has_initial_state", "spec_state_indices",
                  "num_accepted_tokens"):
            t = getattr(sub, k)
            if t is not None:
                idx.append((t, t.cpu().pin_memory()))
    host_out = torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + \
        sum(h.numel() * h.element_size() for _, h in idx)
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for k, t in host_in.items():
            getattr(db, k).copy_(t, non_blocking=True)
        for dev, host in idx:
            dev.copy_(host, non_blocking=True)
        db.run()
        host_out.copy_(db.out, non_blocking=True)

    serial_ms = statistics.median(timed(e2e_step, max(3, steps // 4), flush, stream))

    db2 = to_device(batch, pools=db.pools)
    host_of = dict((id(dv), hv) for dv, hv in idx)
    sets = []
    for d in (db, db2):
        pairs = [(getattr(d, k), host_in[k]) for k in ("x", "a", "b")]
        for sub, hsub in ((d.spec, db.spec), (d.non_spec, db.non_spec)):
            if sub is None:
                continue
            for k in ("query_start_loc", "token_indx", "state_indices", "has_initial_state", "spec_state_indices",
                      "num_accepted_tokens"):
                t = getattr(sub, k)
                if t is not None:
                    pairs.append((t, host_of[id(getattr(hsub, k))]))
        sets.append((d, pairs, torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory()))
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n):
        for i in range(n):
            b = i % 2
            d, pairs, hout = sets[b]
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(done[b])  # step i-2 has finished reading this set's inputs
                for dev, host in pairs:
                    dev.copy_(host, non_blocking=True)
                ready[b].record(h2d_s)
            stream.wait_event(ready[b])
            if i >= 2:
                stream.wait_event(drained[b])  # step i-2's outputs have left this set's buffer
            d.run(stream)
            done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[b])
                hout.copy_(d.out, non_blocking=True)
                drained[b].record(d2h_s)

    # the same kernels back to back without the flush, for comparison with the pipelined number
    for _ in range(3):
        db.run()
    torch.cuda.synchronize()
    n_steady = max(8, steps // 2)
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0e.record(stream)
    for _ in range(n_steady):
        db.run()
    t1e.record(stream)
    torch.cuda.synchronize()
    steady_ms = t0e.elapsed_time(t1e) / n_steady

    pipelined(4)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    n_e2e = max(64, steps // 2)  # long enough that the pipeline's fill and drain do not count
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(h2d_s)
    pipelined(n_e2e)
    d2h_s.wait_stream(stream)
    t_end.record(d2h_s)
    torch.cuda.synchronize()
    return {"ms_per_step": t_start.elapsed_time(t_end) / n_e2e, "serial_ms_per_step": serial_ms,
            "device_ms_per_step_no_flush": steady_ms, "h2d": h2d, "d2h": d2h}


def run_profile(args) -> int:
    """The step of the chosen workload, warmup + steps times back to back on its first index set
    (one pool: the smallest device footprint a profiler has to save and restore)."""
    from gated_deltanet_linear_spec_gb300.device_batch import to_device
    from gated_deltanet_linear_spec_gb300.workloads import with_layouts
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    batch = with_layouts(make_workload(args.workload), qkv_layout=int(args.qkv_layout == "per_khead"),
                         conv_layout=int(args.conv_layout == "per_slot"))
    db = to_device(batch)
    for _ in range(args.warmup + args.steps):
        db.run()
    torch.cuda.synchronize()
    return int(db.status.item() != 0)


def run_sweep(args) -> int:
    """The throughput sweep on one GPU: spec verify at drafts in {1, 2, 4} x batch in {1, 8, 64,
    256, 512} over a 2048-slot pool, then the 8192-token chunked prefill.  Each point prints one
    JSON line: the whole step through gdn_mixed_batch (L2 flushed between steps) and the
    roofline kernel alone."""
    import gated_deltanet_linear_spec_gb300 as gdn
    from gated_deltanet_linear_spec_gb300 import workloads as W
    from gated_deltanet_linear_spec_gb300.device_batch import to_device

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    hbm, bf16 = peaks.get("hbm_gbs") or FALLBACK_HBM_GBS, peaks.get("bf16_tflops") or FALLBACK_BF16_TFLOPS
    points = [(d, b) for d in (1, 2, 4) for b in (1, 8, 64, 256, 512)] + [("prefill", 8192)]
    for d, b in points:
        if d == "prefill":
            batch = W.long_prefill(b)
            name = f"long_prefill: one {b}-token chunked-prefill row, same layer"
        else:
            batch = W.sweep_point(d, b, seed=4 + d * 10 + b)
            name = f"sweep: spec verify, {d} drafts ({d + 1} tokens/row), batch {b}, 2048-slot pool"
        db = to_device(batch)
        alg = algorithmic_bytes(batch)
        steps = max(3, min(args.steps, 400 if d != "prefill" else 20))
        for _ in range(args.warmup):
            db.run()
            flush.zero_()
        torch.cuda.synchronize()
        ms = statistics.median(timed(db.run, steps, flush, stream))
        rows = db.spec if db.spec is not None else db.non_spec
        y = torch.empty((rows.num_tokens, batch.layer.channels), dtype=torch.float32, device="cuda")
        gdn.gdn_conv_update(db.layer, db.params, db.pools, db.x, rows, y, db.status)
        if d == "prefill":
            ws = torch.empty(gdn.gdn_prefill_workspace_bytes(db.layer, rows, rows.num_seqs), dtype=torch.uint8,
                             device="cuda")
            k_ms = statistics.median(timed(lambda: gdn.gdn_chunk_prefill(db.layer, db.params, db.pools, y, db.a, db.b,
                                                                       rows, db.out, ws, status=db.status),
                                         steps, flush, stream))
            roof = {"kernel": "gdn_chunk_prefill", "bound": "tensor", "unit": "TFLOP/s", "peak": bf16,
                    "achieved": prefill_flops(batch) / (k_ms * 1e-3) / 1e12, "launch_ms": k_ms}
        else:
            k_ms = statistics.median(timed(lambda: gdn.gdn_recurrent_step(db.layer, db.params, db.pools, y, db.a, db.b,
                                                                        rows, db.out, db.status),
                                         steps, flush, stream))
            roof = {"kernel": "gdn::recurrent_kernel", "bound": "hbm", "unit": "GB/s", "peak": hbm,
                    "achieved": alg["recurrence"] / (k_ms * 1e-3) / 1e9, "launch_ms": k_ms,
                    "algorithmic_bytes_per_launch": alg["recurrence"]}
        roof["frac"] = roof["achieved"] / roof["peak"]
        T = batch.num_actual_tokens
        line = {"metric": METRIC, "value": T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "sweep": True,
                "config": {"workload": name, "tokens_per_step": T, "l2": "flushed between steps",
                           "hbm_gbs_whole_step": alg["total"] / (ms * 1e-3) / 1e9, "status": int(db.status.item())},
                "roofline": roof}
        print(json.dumps(line), flush=True)
        del db, y
        torch.cuda.empty_cache()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="spec_verify", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--qkv-layout", default="packed", choices=["packed", "per_khead"],
                    help="channel order of x (per_khead: the reorder_input=False projection order)")
    ap.add_argument("--conv-layout", default="rolled", choices=["rolled", "per_slot"],
                    help="spec conv history: rolled at column 0, or one snapshot per spec slot")
    ap.add_argument("--graph", action="store_true", help="time replays of a CUDA graph of the step")
    ap.add_argument("--sweep", action="store_true",
                    help="one line per point of the throughput sweep (drafts x batch, and the long prefill)")
    ap.add_argument("--profile", action="store_true",
                    help="for profilers: warmup + steps plain passes of the first index set, no timing, no output")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.sweep:
        return run_sweep(args)
    if args.profile:
        return run_profile(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    big = args.workload in ("mixed", "long_prefill")
    oracle_heads = (0, 2) if big else None

    if args.impl == "reference":
        if rank != 0:
            return 0
        batch = make_workload(args.workload)
        ref = oracle_tokens_per_s(batch, budget_s=10.0, heads=oracle_heads)
        per_step_s = batch.num_actual_tokens / ref["value"]
        line = {"metric": METRIC, "value": ref["value"], "unit": UNIT, "n_gpus": 0, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": per_step_s * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload_config(args),
                "timing": {"where": "host CPU (the oracle, first index set)", "cores": ref["cores"]},
                "impl": "reference", "cpu_baseline": ref,
                "e2e": {"value": ref["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import gated_deltanet_linear_spec_gb300 as gdn
    from gated_deltanet_linear_spec_gb300.device_batch import to_device
    from gated_deltanet_linear_spec_gb300.workloads import with_layouts

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    clocks = ClockSampler(local_rank)
    batches = [with_layouts(make_workload(args.workload, seed), qkv_layout=int(args.qkv_layout == "per_khead"),
                            conv_layout=int(args.conv_layout == "per_slot")) for seed in INDEX_SETS[args.workload]]
    dbs = [to_device(b) for b in batches]
    algs = [algorithmic_bytes(b) for b in batches]
    batch, db = batches[0], dbs[0]
    T = batch.num_actual_tokens
    assert all(b.num_actual_tokens == T for b in batches)
    nsets = len(dbs)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    steps = args.steps if not big else max(3, args.steps // 40)

    # -------- device-timed steps: the whole path through gdn_mixed_batch, L2 flushed in between,
    #          step i on index set i % nsets
    for i in range(args.warmup):
        dbs[i % nsets].run()
        flush.zero_()
    torch.cuda.synchronize()
    step_fns = [d.run for d in dbs]
    if args.graph:
        graphs = []
        for d in dbs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                d.run()
            graphs.append(g)
        for i in range(args.warmup):
            graphs[i % nsets].replay()
            flush.zero_()
        torch.cuda.synchronize()
        step_fns = [g.replay for g in graphs]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_region0 = time.monotonic()
    step_ms = timed_rotating(step_fns, steps, flush, stream)
    torch.cuda.synchronize()
    clocks.mark(t_region0, time.monotonic())
    if dist:
        dist.barrier()

    # -------- the dominant kernel alone, through the public entry point that launches exactly it
    ys = []
    for d in dbs:
        rows = d.spec if d.spec is not None else d.non_spec
        ys.append(torch.empty((rows.num_tokens, batch.layer.channels), dtype=torch.float32, device="cuda"))

    def conv_fn(d, y):
        rows = d.spec if d.spec is not None else d.non_spec
        return lambda: gdn.gdn_conv_update(d.layer, d.params, d.pools, d.x, rows, y, d.status)

    conv_ms = timed_rotating([conv_fn(d, y) for d, y in zip(dbs, ys)], steps, flush, stream)
    if args.workload == "long_prefill":
        def prefill_fn(d, y):
            rows = d.non_spec
            ws = torch.empty(gdn.gdn_prefill_workspace_bytes(d.layer, rows, rows.num_seqs), dtype=torch.uint8,
                             device="cuda")
            return lambda: gdn.gdn_chunk_prefill(d.layer, d.params, d.pools, y, d.a, d.b, rows, d.out, ws,
                                                 status=d.status)
        kern_ms = timed_rotating([prefill_fn(d, y) for d, y in zip(dbs, ys)], steps, flush, stream)
        flops = [prefill_flops(b) for b in batches]
        peaks = measured_peaks()
        peak = peaks.get("bf16_tflops")
        roof = {"kernel": "gdn chunk_prep_kernel + chunk_scan_kernel (gdn_chunk_prefill)", "bound": "tensor",
                "achieved": per_launch_rate(flops, kern_ms) / 1e12, "peak": peak or FALLBACK_BF16_TFLOPS,
                "peak_source": "measured (bf16 burst)" if peak else "fallback", "unit": "TFLOP/s", "traffic": None,
                "algorithmic_flops_per_launch": statistics.mean(flops), "launch_ms": statistics.median(kern_ms),
                "launch_ms_mean": statistics.mean(kern_ms), "conv_launch_ms": statistics.median(conv_ms)}
    else:
        def rec_fn(d, y):
            rows = d.spec if d.spec is not None else d.non_spec
            return lambda: gdn.gdn_recurrent_step(d.layer, d.params, d.pools, y, d.a, d.b, rows, d.out, d.status)
        rec_ms = timed_rotating([rec_fn(d, y) for d, y in zip(dbs, ys)], steps, flush, stream)
        peaks = measured_peaks()
        peak = peaks.get("hbm_gbs")
        kern_ms, units = rec_ms, [a["recurrence"] for a in algs]
        src = source_hash("gdn_recurrent.cu", "gdn_internal.cuh")
        kname, tkey = "gdn::recurrent_kernel", "recurrent_kernel"
        roof = {"kernel": kname, "bound": "hbm", "achieved": per_launch_rate(units, kern_ms) / 1e9,
                "peak": peak or FALLBACK_HBM_GBS, "peak_source": "measured (copy)" if peak else "fallback",
                "unit": "GB/s", "traffic": recorded_traffic(tkey, args.workload, src),
                "source_hash": src, "algorithmic_bytes_per_launch": statistics.mean(units),
                "launch_ms": statistics.median(kern_ms), "launch_ms_mean": statistics.mean(kern_ms),
                "conv_launch_ms": statistics.median(conv_ms)}
    roof["frac"] = roof["achieved"] / roof["peak"]

    # -------- end to end: pinned host inputs -> device -> gdn_mixed_batch -> host outputs (set 0)
    e2e = end_to_end(db, batch, stream, flush, steps, dist)
    clk = clocks.stop()

    status = int(db.status.item())
    ms, ms_mean = statistics.median(step_ms), statistics.mean(step_ms)
    ms, ms_mean, e2e_ms, e2e_serial_ms, steady_ms = reduce_max_over_ranks(
        [ms, ms_mean, e2e["ms_per_step"], e2e["serial_ms_per_step"], e2e["device_ms_per_step_no_flush"]], dist,
        device="cuda")
    if rank != 0:
        dist.destroy_process_group()
        return 0

    chunked = bool(batch.num_prefills and gdn.gdn_prefill_workspace_bytes(db.layer, db.non_spec, batch.num_prefills))
    launches_per_step = 4 if chunked else 2  # conv, recurrence (+ prep and scan of the prefill rows)
    alg_total = statistics.mean(a["total"] for a in algs)
    line = {
        "metric": METRIC, "value": job_throughput(T, world, ms), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args),
        "timing": {"statistic": "median over the timed steps", "ms_per_step_mean": ms_mean,
                   "l2": "flushed between steps (512 MiB write)",
                   "index_sets": f"step i runs seeded index set i % {nsets} (seeds {list(INDEX_SETS[args.workload])})",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": "cuda graph replay" if args.graph else "eager",
                   "hbm_gbs_whole_step": alg_total / (ms * 1e-3) / 1e9,
                   "algorithmic_bytes_per_step": alg_total, "status": status},
        "roofline": roof,
        "e2e": {"value": job_throughput(T, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e_ms,
                "mode": "pipelined over steps (copies overlap the previous/next step's kernels; no L2 flush: "
                        "the state a step touches exceeds L2); index set 0",
                "serial_ms_per_step": e2e_serial_ms,
                "device_ms_per_step_no_flush": steady_ms},
        "gpu_launches": launches_per_step * steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_tokens_per_s(batch, heads=oracle_heads)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
