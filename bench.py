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
L2_FLUSH_BYTES = 512 << 20


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
                if ssi[0] > 0:
                    conv += (W - 1 + W - 2 + ln) * C * act
            else:
                s = int(sub.state_indices[n])
                hi = 1 if sub.has_initial_state is None else int(sub.has_initial_state[n])
                loads += (s > 0 and hi != 0)
                stores += s > 0
                if s > 0:
                    conv += ((W - 1) * (hi != 0) + (W - 1)) * C * act
    T = batch.num_actual_tokens
    ssm = (loads + stores) * state
    io = T * (C * act + 2 * Hv * act + Hv * dv * act)
    params = C * W * act + 2 * Hv * 4
    rec = ssm + T * (2 * Hv * act + Hv * dv * act)  # what the recurrence kernel must move
    return {"total": ssm + io + conv + params, "ssm": ssm, "recurrence": rec, "conv": conv,
            "state_loads": loads, "state_stores": stores}


# ------------------------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)

def oracle_tokens_per_s(batch, budget_s: float = 12.0) -> dict:
    from tests.oracle_run import np_act, run_oracle
    cores = len(os.sched_getaffinity(0))
    conv_pool, ssm_pool = np_act(batch.conv_pool), np_act(batch.ssm_pool)  # copied once, outside the timing
    reps, el = 0, 0.0
    while el < budget_s and reps < 50:
        t0 = time.perf_counter()
        run_oracle(batch, nthreads=cores, conv_pool=conv_pool, ssm_pool=ssm_pool)
        el += time.perf_counter() - t0
        reps += 1
    return {"value": reps * batch.num_actual_tokens / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the full workload ({batch.num_actual_tokens} verify tokens, all 32 heads) repeated "
                      f"{reps}x, {el:.1f} s of CPU time on {cores} threads"}


# ------------------------------------------------------------------------------------------

def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from gated_deltanet_linear_spec_gb300 import workloads

    if args.impl == "reference":
        if rank != 0:
            return 0
        batch = workloads.spec_verify()
        ref = oracle_tokens_per_s(batch, budget_s=10.0)
        per_step_s = batch.num_actual_tokens / ref["value"]
        line = {"metric": METRIC, "value": ref["value"], "unit": UNIT, "n_gpus": 0, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": per_step_s * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOAD}, "impl": "reference", "cpu_baseline": ref,
                "e2e": {"value": ref["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import gated_deltanet_linear_spec_gb300 as gdn
    from gated_deltanet_linear_spec_gb300.device_batch import to_device

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    batch = workloads.spec_verify()
    db = to_device(batch)
    alg = algorithmic_bytes(batch)
    T = batch.num_actual_tokens
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    # -------- device-timed steps (the whole path through gdn_mixed_batch)
    for _ in range(args.warmup):
        db.run()
        flush.zero_()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        ev[i][0].record(stream)
        db.run()
        ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # -------- the recurrence kernel alone (same kernels, split into the two public calls)
    y = torch.empty((T, batch.layer.channels), dtype=torch.float32, device="cuda")
    rec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    conv_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for i in range(args.steps):
        conv_ev[i][0].record(stream)
        gdn.gdn_conv_update(db.layer, db.params, db.pools, db.x, db.spec, y, db.status)
        conv_ev[i][1].record(stream)
        rec_ev[i][0].record(stream)
        gdn.gdn_recurrent_step(db.layer, db.params, db.pools, y, db.a, db.b, db.spec, db.out, db.status)
        rec_ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    clk = clocks.stop()
    rec_ms = statistics.mean(a.elapsed_time(b) for a, b in rec_ev)
    conv_ms = statistics.mean(a.elapsed_time(b) for a, b in conv_ev)

    # -------- end to end: pinned host inputs -> device -> gdn_mixed_batch -> host outputs
    host_in = {k: getattr(db, k).cpu().pin_memory() for k in ("x", "a", "b")}
    idx_names = ("query_start_loc", "spec_state_indices", "num_accepted_tokens")
    host_idx = {k: getattr(db.spec, k).cpu().pin_memory() for k in idx_names}
    host_out = torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(host_in.values()) + list(host_idx.values()))
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(10, args.steps // 4)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        e2e_ev[i][0].record(stream)
        for k, t in host_in.items():
            getattr(db, k).copy_(t, non_blocking=True)
        for k, t in host_idx.items():
            getattr(db.spec, k).copy_(t, non_blocking=True)
        db.run()
        host_out.copy_(db.out, non_blocking=True)
        e2e_ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_ev)

    status = int(db.status.item())
    ms = statistics.mean(step_ms)
    if dist:
        t = torch.tensor([ms, e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, e2e_ms = float(t[0]), float(t[1])
    if rank != 0:
        dist.destroy_process_group()
        return 0

    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    achieved = alg["recurrence"] / (rec_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": world * T / (ms * 1e-3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "flushed between steps (512 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "hbm_gbs_whole_step": alg["total"] / (ms * 1e-3) / 1e9,
                   "algorithmic_bytes_per_step": alg["total"], "status": status},
        "roofline": {"kernel": "gdn::recurrent_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": alg["recurrence"], "launch_ms": rec_ms,
                     "conv_launch_ms": conv_ms},
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_tokens_per_s(batch)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
