#!/usr/bin/env python
"""Benchmark of the verification hot path on the 64-request token-level workload.

Workload: 64 requests x 5 drafted positions (+ 1 bonus row), V = 151936, bf16 logits (target
N(0, 3^2) plus a Zipf(1.1) log-prior, draft = target + N(0, 1)), drafts sampled from q.  One step =
one spec_verify_token call over the whole batch (row statistics, acceptance walk, correction /
bonus races).  Inputs (213.9 MB) are larger than L2, and L2 is also flushed before every timed step
(a 512 MB write, then a 256 MB read so that no dirty flush lines remain); steps are timed with CUDA
events on the launching stream.

Printed: one JSON line (rank 0).  `value` is logit GB/s over the algorithmic bytes of a step
(every drafted target and draft row and every request's bonus row, once); `positions_per_s` is
drafted positions verified per second.  Supplementary rows time the other calls of the library on
their own workloads.

--impl reference times the CPU oracle (the plain double-precision restatement of the method) on the
host cores, on a bounded sample of the same workload, under the same metric.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify logits GB/s (% of GB300 HBM peak) and drafted positions verified/sec"
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the supplementary rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["markov", "schedule", "block", "lmhead", "round"],
                    default=None,
                    help="time one supplementary row alone and print it (profiling runs)")
    ap.add_argument("--markov-positions", type=int, default=None,
                    help="with --only markov: draft this many positions instead of 16")
    return ap.parse_args()


# ---- environment helpers ---------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_digest(files):
    """Digest of the CUDA sources a kernel is built from; a stored ncu traffic figure is used only
    if it was taken on the same sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_token_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_counter(kernel_key, field):
    """A per-launch ncu counter of `kernel_key` (profiles/traffic.json) if taken on these sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    ent = data.get(kernel_key)
    if not ent or ent.get("source_digest") != source_digest(ent.get("sources", [])):
        return None
    return ent.get(field)


def stored_traffic(kernel_key):
    """Per-launch DRAM bytes of `kernel_key` from profiles/traffic.json if taken on these sources."""
    return stored_counter(kernel_key, "dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- workload -----------------------------------------------------------------------------------

def token_workload(device):
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    w = synth.TOKEN_LARGE
    inp = synth.token_inputs(w, device=device)
    tokens = sv.spec_sample_draft(inp["draft"], inp["draft_row0"], inp["draft_len"], w.gamma,
                                  w.seed)
    torch.cuda.synchronize()
    return w, inp, tokens


def necessary_bytes(w, accepted_len, esize):
    """Drafted target + draft rows of every request, plus the bonus row where all were kept."""
    n_bonus = int((accepted_len == w.gamma).sum())
    return (2 * w.B * w.gamma + n_bonus) * w.V * esize, n_bonus


def make_flush(dev):
    """L2 flush between timed calls: a 512 MB write evicts every line the previous call left in
    L2, and a 256 MB read of the same buffer then evicts the flush's own dirty lines, so that the
    timed call neither finds its inputs in L2 nor pays for writing the flush buffer back."""
    import torch
    buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    head = buf[: L2_FLUSH_BYTES // 2]

    def flush():
        buf.fill_(1)
        head.sum()
    return flush


def max_over_ranks(x, world, device):
    """The largest of every rank's x (each rank passes its own); x itself on a single rank."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, steps, world, max_time):
    """Units per second over all ranks: every rank (replica) processes units_per_rank_step units
    per step, and the job takes as long as its slowest rank."""
    return units_per_rank_step * world * steps / max_time


def time_calls(fn, steps, warmup, flush, stream):
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    return times


def bench_token(args, rank, world, peaks, peak_src):
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    w, inp, tokens = token_workload(dev)
    esize = inp["target"].element_size()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SV_BF16), dev)
    flush = make_flush(dev)
    holder = {}

    def step():
        holder["out"] = sv.spec_verify_token(inp["target"], inp["draft"], inp["target_row0"],
                                             inp["draft_row0"], inp["draft_len"], w.gamma,
                                             tokens, w.seed, status=status, workspace=ws)

    with ClockSampler(dev.index) as clocks:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        times = time_calls(step, args.steps, args.warmup, flush, stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    assert int(status.item()) == 0, sv.status_string(int(status.item()))
    # per-kernel durations (CUDA events the library records between its kernels on this stream)
    sv.sv_profile_enable(True)
    parts = []
    for _ in range(max(3, args.steps // 2)):
        flush()
        step()
        parts.append(sv.sv_profile_read())
    sv.sv_profile_enable(False)
    kernel_ms = [sum(p[k] for p in parts) / len(parts) for k in range(3)]
    acc = holder["out"]["accepted_len"].cpu()
    nbytes, n_bonus = necessary_bytes(w, acc, esize)
    all_rows_bytes = (2 * w.B * w.gamma + w.B) * w.V * esize
    t_mean = sum(times) / len(times)
    total_time = max_over_ranks(sum(times), world, dev)
    res = {
        "w": w, "times": times, "t_mean": t_mean, "total_time": total_time,
        "bytes": nbytes, "all_rows_bytes": all_rows_bytes, "n_bonus": n_bonus,
        "positions": w.B * w.gamma, "clocks": clocks.summary(), "inp": inp, "tokens": tokens,
        "accept_mean": float(acc.float().mean()),
        "kernel_ms": kernel_ms,
    }
    return res


def bench_e2e(w, inp, tokens, steps, warmup):
    """The same call fed from pinned host buffers: H2D of the step's logits and layout, verify,
    D2H of the results, all inside the timed region."""
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    dev = inp["target"].device
    stream = torch.cuda.current_stream()
    host = {k: inp[k].cpu().pin_memory() for k in ("target", "draft", "target_row0", "draft_row0",
                                                     "draft_len")}
    host["tokens"] = tokens.cpu().pin_memory()
    devb = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SV_BF16), dev)
    out_host = {"accepted_len": torch.empty(w.B, dtype=torch.int32).pin_memory(),
                "out_tokens": torch.empty((w.B, w.gamma + 1), dtype=torch.int32).pin_memory(),
                "correction": torch.empty(w.B, dtype=torch.int32).pin_memory()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in out_host.values())

    def step():
        for k, v in host.items():
            devb[k].copy_(v, non_blocking=True)
        out = sv.spec_verify_token(devb["target"], devb["draft"], devb["target_row0"],
                                   devb["draft_row0"], devb["draft_len"], w.gamma,
                                   devb["tokens"], w.seed, status=status, workspace=ws)
        for k in out_host:
            out_host[k].copy_(out[k], non_blocking=True)

    times = time_calls(step, steps, warmup, lambda: None, stream)
    return sum(times) / len(times), h2d, d2h, out_host["accepted_len"].clone()


# ---- CPU oracle (baseline and reference arm) --------------------------------------------------

def oracle_sample(w, inp, tokens, target_seconds=12.0, threads=None):
    """Times the oracle on whole requests of the workload, threads over requests on `threads`
    host cores (all of them by default), repeating the request set until about `target_seconds`
    of CPU work is done."""
    import numpy as np
    import oracle
    oracle.build()
    t = inp["target"].float().cpu().numpy()
    d = inp["draft"].float().cpu().numpy()
    tok = tokens.cpu().numpy()
    lay = {k: inp[k].cpu().numpy() for k in ("target_row0", "draft_row0", "draft_len")}
    V, G = w.V, w.gamma
    cores = threads or os.cpu_count() or 1

    def one(r):
        t0 = lay["target_row0"][r]
        d0 = lay["draft_row0"][r]
        res, _ = oracle.verify_token_request(t[t0:t0 + G + 1], d[d0:d0 + G], tok[d0:d0 + G],
                                             w.seed, r)
        return res.accepted_len

    # one probe request to size the sample
    p0 = time.perf_counter()
    one(0)
    per_req = time.perf_counter() - p0
    n_req = max(cores, int(target_seconds / max(per_req, 1e-4)))
    reqs = [r % w.B for r in range(n_req)]
    s0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        accs = list(ex.map(one, reqs))
    wall = time.perf_counter() - s0
    accs = np.array(accs)
    n_bonus = int((accs == G).sum())
    esize = inp["target"].element_size()
    nbytes = (2 * G * n_req + n_bonus) * V * esize
    alg = (2 * G + 1) * n_req * V * esize  # every row of the sampled requests, bonus included
    return {"gbs": alg / wall / 1e9, "gbs_read": nbytes / wall / 1e9,
            "positions_per_s": G * n_req / wall, "cores": cores,
            "wall_s": wall, "requests": n_req,
            "sample": f"{n_req} whole requests of the workload (request set repeated), "
                      f"{G} drafted positions each, V={V}, "
                      + ("threads over requests" if cores > 1 else "one thread")}


# ---- supplementary rows ---------------------------------------------------------------------------

def bench_rows(steps, warmup):
    import numpy as np
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    flush = make_flush(dev)
    rows = {}
    rows["block_verify_128x7_V129280_bf16"] = bench_block(steps, warmup, flush, stream)

    # scheduler, 512 requests x 16 positions
    sw = synth.SCHEDULE
    si = synth.schedule_inputs(sw)
    c = torch.from_numpy(si["cond_accept"]).to(dev)
    ml = torch.from_numpy(si["max_len"]).to(dev)
    sps = torch.from_numpy(si["sps"]).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sws = sv.workspace(sv.dspark_schedule_workspace_bytes(sw.N, sw.K), dev)
    sched = {}

    def sch():
        sched["o"] = sv.dspark_schedule(c, ml, sps, si["B_max"], status=status, workspace=sws)
    t = time_calls(sch, steps, warmup, flush, stream)  # the flush keeps the GPU ahead of the host
    rows["schedule_512x16"] = {"us": sum(t) / len(t) * 1e6,
                               "kernel_us": schedule_kernel_us(sch, steps, flush),
                               "total_rows": int(sched["o"]["total_rows"].item()),
                               "status": int(status.item())}

    # the best-budget rule on the same inputs, and one per-position acceptance update
    def sch_best():
        sched["o"] = sv.dspark_schedule(c, ml, sps, si["B_max"], status=status, workspace=sws,
                                        rule=sv.SV_STOP_ARGMAX)
    t = time_calls(sch_best, steps, warmup, flush, stream)
    rows["schedule_best_budget_512x16"] = {
        "us": sum(t) / len(t) * 1e6, "total_rows": int(sched["o"]["total_rows"].item()),
        "status": int(status.item())}

    def sch_depth():
        sched["o"] = sv.dspark_schedule(c, ml, sps, si["B_max"], status=status, workspace=sws,
                                        rule=sv.SV_STOP_FIXED_DEPTH)
    t = time_calls(sch_depth, steps, warmup, flush, stream)
    rows["schedule_fixed_depth_512x16"] = {
        "us": sum(t) / len(t) * 1e6, "total_rows": int(sched["o"]["total_rows"].item()),
        "status": int(status.item())}
    sch_best()  # the acceptance update below reads the best-budget selection
    sel = sched["o"]["sel_len"]
    acc = torch.minimum(sel, torch.arange(sw.N, device=dev, dtype=torch.int32) % 5)
    trials = torch.zeros(sw.K, dtype=torch.float64, device=dev)
    accepts = torch.zeros(sw.K, dtype=torch.float64, device=dev)
    cond_out = torch.empty((sw.N, sw.K), dtype=torch.float32, device=dev)
    alpha = torch.empty(sw.K, dtype=torch.float32, device=dev)

    def upd():
        sv.dspark_acceptance_update(sel, acc, trials, accepts, decay=0.99, alpha=alpha,
                                    cond_accept_out=cond_out, status=status)
    t = time_calls(upd, steps, warmup, flush, stream)
    rows["acceptance_update_512x16"] = {"us": sum(t) / len(t) * 1e6,
                                        "status": int(status.item())}

    # temperature fit of the confidence head over 64 verified rounds of 512 requests x 16
    rng = np.random.default_rng(5)
    n_cal = 64 * sw.N
    scores = torch.from_numpy(rng.normal(0.0, 2.0, (n_cal, sw.K)).astype(np.float32)).to(dev)
    cal_sel = torch.full((n_cal,), sw.K, dtype=torch.int32, device=dev)
    cal_acc = torch.from_numpy((rng.geometric(0.3, n_cal) - 1).clip(0, sw.K).astype(np.int32)).to(dev)
    fit = {}

    def sts():
        fit["o"] = sv.dspark_sts_fit(scores, cal_sel, cal_acc, status=status)
    t = time_calls(sts, max(3, steps // 3), warmup, flush, stream)
    rows["sts_fit_32768x16"] = {"us": sum(t) / len(t) * 1e6, "newton_steps": 30,
                                "status": int(status.item())}

    rows["scheduled_round_512x16_V129280_bf16"] = bench_round(steps, warmup, flush, stream)
    rows["markov_draft_256x16_V151936_R256"] = bench_markov(steps, warmup, flush, stream)
    rows["lmhead_verify_64x5_V151936_H2560_bf16"] = bench_lmhead(steps, warmup, flush, stream)
    return rows


def bench_round(steps, warmup, flush, stream):
    """A scheduled round: the scheduler over 512 requests x 16 positions, then token verification
    of the selected prefixes (V = 129280, bf16)."""
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    sw = synth.SCHEDULE
    si = synth.schedule_inputs(sw)
    c = torch.from_numpy(si["cond_accept"]).to(dev)
    ml = torch.from_numpy(si["max_len"]).to(dev)
    sps = torch.from_numpy(si["sps"]).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sws = sv.workspace(sv.dspark_schedule_workspace_bytes(sw.N, sw.K), dev)
    # scheduled round: schedule, then verify the selected prefixes (V = 129280)
    vw = synth.SCHEDULED_VERIFY
    vin = synth.token_inputs(vw, device=dev)
    vt = sv.spec_sample_draft(vin["draft"], vin["draft_row0"], vin["draft_len"], vw.gamma,
                              vw.seed)
    ws2 = sv.workspace(sv.spec_verify_workspace_bytes(vw.B, vw.gamma, vw.V, sv.SV_BF16), dev)
    rnd = {}

    def round_():
        s = sv.dspark_schedule(c, ml, sps, si["B_max"], status=status, workspace=sws)
        rnd["o"] = sv.spec_verify_token(vin["target"], vin["draft"], vin["target_row0"],
                                        vin["draft_row0"], s["sel_len"], vw.gamma, vt, vw.seed,
                                        status=status, workspace=ws2)
        rnd["s"] = s
    t = time_calls(round_, steps, warmup, flush, stream)
    # the verify call's kernels (stream, race), from the library's events (the last call records)
    sv.sv_profile_enable(True)
    parts = []
    for _ in range(max(3, steps // 2)):
        flush()
        round_()
        parts.append(sv.sv_profile_read())
    sv.sv_profile_enable(False)
    vkms = [sum(q[k] for q in parts) / len(parts) for k in range(3)]
    sel = rnd["s"]["sel_len"].cpu()
    acc = rnd["o"]["accepted_len"].cpu()
    n_bonus = int((acc == sel).sum())
    nb = (2 * int(sel.sum()) + n_bonus) * vw.V * 2
    tm = sum(t) / len(t)
    row = {
        "ms": tm * 1e3, "GB_s": nb / tm / 1e9, "positions_per_s": int(sel.sum()) / tm,
        "verified_rows": int(rnd["s"]["total_rows"].item()),
        "verify_kernel_ms": {"stream": round(vkms[0], 4), "race_with_decide": round(vkms[2], 4)},
        "status": int(status.item())}
    del vin, vt
    return row


def bench_schedule(steps, warmup):
    """The scheduler alone on the 512 x 16 workload, each call behind the L2 flush so that the host
    stays ahead of the GPU."""
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = make_flush(dev)
    sw = synth.SCHEDULE
    si = synth.schedule_inputs(sw)
    c = torch.from_numpy(si["cond_accept"]).to(dev)
    ml = torch.from_numpy(si["max_len"]).to(dev)
    sps = torch.from_numpy(si["sps"]).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.dspark_schedule_workspace_bytes(sw.N, sw.K), dev)
    out = {}

    def sch():
        out["o"] = sv.dspark_schedule(c, ml, sps, si["B_max"], status=status, workspace=ws)
    t = time_calls(sch, steps, warmup, flush, torch.cuda.current_stream())
    return {"workload": f"{sw.N} requests x {sw.K} positions, B_max={sw.B_max}",
            "us": sum(t) / len(t) * 1e6, "kernel_us": schedule_kernel_us(sch, steps, flush),
            "total_rows": int(out["o"]["total_rows"].item()), "status": int(status.item())}


def schedule_kernel_us(call, steps, flush):
    """Device durations of the scheduler's two kernels (rank, admit), from the CUDA events the
    library records around them when profiling is on."""
    import speculative_decoding_verification_token_gb300 as sv
    sv.sv_profile_enable(True)
    parts = []
    for _ in range(max(3, steps // 2)):
        flush()
        call()
        parts.append(sv.sv_profile_read())
    sv.sv_profile_enable(False)
    return {"rank": round(sum(q[0] for q in parts) / len(parts) * 1e3, 2),
            "admit": round(sum(q[2] for q in parts) / len(parts) * 1e3, 2)}


def bench_block(steps, warmup, flush, stream):
    """Block verification, 128 requests x 7 drafted positions, V = 129280 bf16."""
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    w = synth.BLOCK_LARGE
    inp = synth.token_inputs(w, device=dev)
    tokens = sv.spec_sample_draft(inp["draft"], inp["draft_row0"], inp["draft_len"], w.gamma,
                                  w.seed)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SV_BF16), dev)
    holder = {}

    def blk(want_rows):
        def call():
            holder["o"] = sv.spec_verify_block(inp["target"], inp["draft"], inp["target_row0"],
                                               inp["draft_row0"], inp["draft_len"], w.gamma,
                                               tokens, w.seed, want_rows=want_rows,
                                               status=status, workspace=ws)
        return call
    # the call a user makes for the tokens alone (no per-row outputs), then the same call with
    # every running ratio and threshold written (every residual mass computed)
    t = time_calls(blk(False), steps, warmup, flush, stream)
    st_tok = int(status.item())
    acc = holder["o"]["accepted_len"].cpu()
    t_rows = time_calls(blk(True), steps, warmup, flush, stream)
    # device durations of the tokens-only call's kernels: the row-statistics stream, the prep and
    # residual-mass kernels, the decision and race (events between them: serialised)
    sv.sv_profile_enable(True)
    parts = []
    call = blk(False)
    for _ in range(max(3, steps // 2)):
        flush()
        call()
        parts.append(sv.sv_profile_read())
    sv.sv_profile_enable(False)
    kms = [sum(q[k] for q in parts) / len(parts) for k in range(3)]
    n_bonus = int((acc == w.gamma).sum())
    nb = (2 * w.B * w.gamma + n_bonus) * w.V * 2
    tm = sum(t) / len(t)
    tr = sum(t_rows) / len(t_rows)
    return {
        "ms": tm * 1e3, "GB_s": nb / tm / 1e9, "positions_per_s": w.B * w.gamma / tm,
        "ms_with_row_outputs": tr * 1e3, "GB_s_with_row_outputs": nb / tr / 1e9,
        "kernel_ms": {"stream": round(kms[0], 4), "prep_and_residuals": round(kms[1], 4),
                      "decide_and_race": round(kms[2], 4)},
        "mean_accepted": float(acc.float().mean()),
        "status": st_tok or int(status.item())}


def bench_markov(steps, warmup, flush, stream, positions=None):
    """DSpark Markov-head drafting: 256 requests x 16 positions, V = 151936, R = 256, bf16.  One
    call drafts every position (16 position kernels + 16 select kernels).  Algorithmic bytes per
    call: the backbone read and z written once (2 x 1.245 GB) plus Wt read once per position
    (77.8 MB, usually from L2 after the first); FLOPs: 2 B R V per position."""
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    w = synth.MARKOV
    if positions is not None:
        w = dataclasses.replace(w, K=positions)
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = synth.markov_inputs(w, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.dspark_markov_workspace_bytes(w.B, w.K, w.V, w.R), dev)
    holder = {}

    def call():
        holder["o"] = sv.dspark_markov_draft(inp["backbone"], inp["U"], inp["Wt"], inp["anchor"],
                                             inp["scores"], inp["T"], w.seed, status=status,
                                             workspace=ws)
    t = time_calls(call, steps, warmup, flush, stream)
    assert int(status.item()) == 0, sv.status_string(int(status.item()))
    sv.sv_profile_enable(True)
    parts = []
    for _ in range(max(3, steps // 2)):
        flush()
        call()
        parts.append(sv.sv_profile_read())
    sv.sv_profile_enable(False)
    pos_ms = sum(p[0] for p in parts) / len(parts)   # position kernel of k = 1
    sel_ms = sum(p[1] for p in parts) / len(parts)   # its select kernel
    tm = sum(t) / len(t)
    elems = w.B * w.K * w.V
    # algorithmic bytes: the backbone read and z written once, W read once per call
    bytes_call = 2 * elems * 2 + w.V * w.R * 2
    # bytes the kernels move when W is re-read at every position (it does not stay in L2)
    bytes_moved = 2 * elems * 2 + w.K * w.V * w.R * 2
    flops_call = 2.0 * w.B * w.R * w.V * w.K
    # one position kernel: its backbone and z rows and one read of W
    pos_bytes = 2 * w.B * w.V * 2 + w.V * w.R * 2
    peaks, _ = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    tf = float(peaks["bf16_tflops"])
    # instruction issue, the bound of the epilogue: warp instructions per position kernel (ncu,
    # stored with its sources' digest) over the kernel's time, against one warp instruction per
    # scheduler and clock (152 SMs x 4 schedulers x the maximum SM clock)
    inst = stored_counter("markov_position_256_V151936_R256", "warp_instructions_per_launch")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    issue_peak = sms * 4 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
    alu = None
    if inst:
        achieved = inst / (pos_ms * 1e-3)
        alu = {"bound": "alu", "achieved": achieved, "peak": issue_peak,
               "unit": "warp instructions/s", "frac": achieved / issue_peak,
               "warp_instructions_per_position_kernel": inst,
               "peak_note": "SMs x 4 schedulers x one warp instruction per clock at the maximum "
                            "SM clock"}
    return {
        "workload": f"{w.B} requests x {w.K} positions, V={w.V}, R={w.R}, bf16",
        "alu_roofline": alu,
        "ms": tm * 1e3, "ms_median": statistics.median(t) * 1e3,
        "drafted_positions_per_s": w.B * w.K / tm,
        "algorithmic_bytes_per_call": bytes_call,
        "bytes_moved_per_call_W_per_position": bytes_moved,
        "GB_s": bytes_call / tm / 1e9, "hbm_frac_of_measured": bytes_call / tm / 1e9 / hbm,
        "TFLOP_s": flops_call / tm / 1e12, "tensor_frac_of_measured": flops_call / tm / 1e12 / tf,
        "sampled_elements_per_s": elems / tm,
        "position_kernel_ms": pos_ms, "select_kernel_ms": sel_ms,
        "position_kernel_GB_s": pos_bytes / (pos_ms * 1e-3) / 1e9,
        "position_kernel_TFLOP_s": flops_call / w.K / (pos_ms * 1e-3) / 1e12,
        "kernel_ms_note": "position and select kernel times from a separate run with CUDA events "
                          "between the library's kernels (serialised)",
        "launches_per_call": 2 * w.K, "status": int(status.item())}


def bench_lmhead(steps, warmup, flush, stream):
    """Verification from hidden states: 64 requests x 5 drafted positions, V = 151936, H = 2560,
    bf16 hidden rows and output projection (spec_verify_lmhead).  Algorithmic work per call: the
    logits of the B (2 gamma + 1) target and draft rows, 2 Q H V FLOPs ("How much does a token
    cost", "The Role of Arithmetic Intensity"), and one read of W plus the hidden rows."""
    import torch
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import synth
    w = synth.LMHEAD
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = synth.lmhead_inputs(w, device=dev)
    # drafted tokens (setup, untimed): the draft's logits through W, sampled by the library
    dlog = inp["draft_hidden"].float() @ inp["W"].float().t()
    tokens = sv.spec_sample_draft(dlog, inp["draft_row0"], inp["draft_len"], w.gamma, w.seed)
    del dlog
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.spec_verify_lmhead_workspace_bytes(w.B, w.gamma, w.V, w.H), dev)
    holder = {}

    def call():
        holder["o"] = sv.spec_verify_lmhead(inp["target_hidden"], inp["draft_hidden"], inp["W"],
                                            inp["target_row0"], inp["draft_row0"],
                                            inp["draft_len"], w.gamma, tokens, w.seed,
                                            status=status, workspace=ws)
    t = time_calls(call, steps, warmup, flush, stream)
    st = int(status.item())
    out = holder["o"]
    sv.sv_profile_enable(True)
    parts = []
    for _ in range(max(3, steps // 2)):
        flush()
        call()
        parts.append(sv.sv_profile_read())
    sv.sv_profile_enable(False)
    kms = [sum(q[k] for q in parts) / len(parts) for k in range(3)]
    # context only, not part of the path: the same logits as one cuBLAS bf16 GEMM (bf16 output),
    # the first step of a pipeline that stores logits and verifies them afterwards
    rows = w.B * (2 * w.gamma + 1)
    hidden = torch.randn((rows, w.H), device=dev, dtype=torch.bfloat16)
    Wt = inp["W"].t()
    t_gemm = time_calls(lambda: hidden @ Wt, steps, warmup, flush, stream)
    del hidden
    tm = sum(t) / len(t)
    flops = 2.0 * rows * w.H * w.V
    slots = -(-w.B * 2 * (w.gamma + 1) // 128) * 128
    w_bytes = w.V * w.H * 2
    peaks, _ = measured_peaks()
    tf = float(peaks["bf16_tflops"])
    return {
        "workload": f"{w.B} requests x {w.gamma} positions, V={w.V}, H={w.H}, bf16",
        "ms": tm * 1e3, "ms_median": statistics.median(t) * 1e3,
        "positions_per_s": w.B * w.gamma / tm,
        "algorithmic_flops_per_call": flops,
        "TFLOP_s": flops / tm / 1e12, "tensor_frac_of_measured": flops / tm / 1e12 / tf,
        "computed_flops_per_call": 2.0 * slots * w.H * w.V,
        "W_bytes_per_call": w_bytes, "W_GB_s": w_bytes / tm / 1e9,
        "kernel_ms": {"gather_and_statistics_gemm": round(kms[0], 4),
                      "decide": round(kms[1], 4), "race_gemm_and_finish": round(kms[2], 4)},
        "kernel_ms_note": "from a separate run with CUDA events between the library's kernels "
                          "(serialised, no programmatic overlap)",
        "recomputed_requests": int(out["recomputed"].item()),
        "mean_accepted": float(out["accepted_len"].float().mean()),
        "context_cublas_logits_gemm_bf16_out_ms": sum(t_gemm) / len(t_gemm) * 1e3,
        "status": st}


# ---- main ----------------------------------------------------------------------------------------

def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    peaks, peak_src = measured_peaks()

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    torch.cuda.set_device(local_rank)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
        __graft_entry__.build()
    if args.only == "markov":
        row = bench_markov(args.steps, args.warmup, make_flush(torch.device("cuda")),
                           torch.cuda.current_stream(), args.markov_positions)
        print(json.dumps({"row": "markov_draft", **row}))
        return
    if args.only == "block":
        row = bench_block(args.steps, args.warmup, make_flush(torch.device("cuda")),
                          torch.cuda.current_stream())
        print(json.dumps({"row": "block_verify", **row}))
        return
    if args.only == "schedule":
        row = bench_schedule(args.steps, args.warmup)
        print(json.dumps({"row": "schedule", **row}))
        return
    if args.only == "round":
        row = bench_round(args.steps, args.warmup, make_flush(torch.device("cuda")),
                          torch.cuda.current_stream())
        print(json.dumps({"row": "scheduled_round", **row}))
        return
    if args.only == "lmhead":
        row = bench_lmhead(args.steps, args.warmup, make_flush(torch.device("cuda")),
                           torch.cuda.current_stream())
        print(json.dumps({"row": "lmhead_verify", **row}))
        return

    res = bench_token(args, rank, world, peaks, peak_src)
    w = res["w"]
    esize = 2
    alg = res["all_rows_bytes"]  # every target and draft row once, each bonus row included
    value = whole_job_rate(alg, args.steps, world, res["total_time"]) / 1e9
    pos_s = whole_job_rate(res["positions"], args.steps, world, res["total_time"])
    hbm = float(peaks["hbm_gbs"])
    t_med = statistics.median(res["times"])
    stream_s = res["kernel_ms"][0] * 1e-3
    stream_bytes = w.B * w.gamma * 2 * w.V * esize  # the row pairs the stream kernel reads
    achieved = stream_bytes / stream_s / 1e9
    e2e_t, h2d, d2h, _ = bench_e2e(w, res["inp"], res["tokens"], max(3, args.steps // 3),
                                   max(3, args.warmup))
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["t_mean"] * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",  # the arithmetic (softmax statistics, ratios, race keys); logits are bf16
        "data": "synthetic",
        "config": token_config(w, world),
        "ms_per_step_median": round(t_med * 1e3, 4),
        "value_median": round(alg / t_med / 1e9, 1),
        "positions_per_s": round(pos_s, 1),
        "bytes_per_step": alg,
        "bytes_definition": "algorithmic: every drafted target and draft row and every request's "
                            "bonus row, once ((2 gamma + 1) B V 2 bytes)",
        "bytes_read_per_step": res["bytes"],
        "bonus_rows_read": res["n_bonus"],
        "call_hbm_frac": {"of_measured": round(alg / res["t_mean"] / 1e9 / hbm, 4),
                          "of_nominal_8000": round(alg / res["t_mean"] / 1e9 / 8000.0, 4),
                          "median_of_measured": round(alg / t_med / 1e9 / hbm, 4)},
        "kernel_ms": {"stream": round(res["kernel_ms"][0], 4),
                      "race_with_decide": round(res["kernel_ms"][1] + res["kernel_ms"][2], 4),
                      "note": "from separate calls with CUDA events recorded between the "
                              "library's kernels: serialised, so their sum exceeds the step"},
        "mean_accepted_len": round(res["accept_mean"], 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "frac_of_nominal_8000": round(achieved / 8000.0, 4),
                     "traffic": stored_traffic("token_verify_64x5_V151936"),
                     "kernel": "stream_kernel (row statistics of every drafted row pair)",
                     "bytes_per_launch": stream_bytes,
                     "peak_source": peak_src},
        "e2e": {"value": round(alg / e2e_t / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_t * 1e3, 4)},
        "gpu_launches": 2 * args.steps,  # stream + race (which decides) per step
        "clocks": res["clocks"],
    }
    if not args.no_rows and rank == 0:
        line["rows"] = bench_rows(max(5, args.steps // 3), max(3, args.warmup))
    if not args.no_cpu_baseline and rank == 0:
        cpu = oracle_sample(w, res["inp"], res["tokens"])
        one = oracle_sample(w, res["inp"], res["tokens"], target_seconds=6.0, threads=1)
        line["cpu_baseline"] = {"value": round(cpu["gbs"], 4), "unit": "GB/s",
                                "cores": cpu["cores"], "kind": "oracle",
                                "sample": cpu["sample"],
                                "positions_per_s": round(cpu["positions_per_s"], 2),
                                "single_thread": {"value": round(one["gbs"], 4), "unit": "GB/s",
                                                  "cores": 1, "sample": one["sample"],
                                                  "positions_per_s":
                                                      round(one["positions_per_s"], 2)}}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def token_config(w, world):
    """The workload both arms report (the reference arm times the CPU oracle on samples of it)."""
    return {"workload": "token-level verify, 64 requests x 5 drafted positions + bonus, "
                        "V=151936, bf16 logits (target N(0,9) + Zipf(1.1) prior, draft = "
                        "target + N(0,1)), drafts sampled from q",
            "B": w.B, "gamma": w.gamma, "V": w.V,
            "l2": "inputs (213.9 MB) larger than L2, and L2 flushed before every step "
                  "by a 512 MB write followed by a 256 MB read (no dirty flush lines "
                  "left to write back inside the timed region)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, rank, world):
    """CPU oracle under the same metric: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    import torch
    from speculative_decoding_verification_token_gb300 import synth
    import oracle
    oracle.build()
    w = synth.TOKEN_LARGE
    inp = synth.token_inputs(w, device="cpu")
    t = inp["target"].float().numpy()
    d = inp["draft"].float().numpy()
    lay = {k: inp[k].numpy() for k in ("target_row0", "draft_row0", "draft_len")}
    st, tokens = oracle.sample_draft_batch(d, w.V, w.V, lay["draft_row0"], lay["draft_len"], w.B,
                                           w.seed)
    cores = os.cpu_count() or 1
    n_req = min(w.B, max(cores, 16))
    import numpy as np

    def one(r):
        t0, d0 = lay["target_row0"][r], lay["draft_row0"][r]
        res, _ = oracle.verify_token_request(t[t0:t0 + w.gamma + 1], d[d0:d0 + w.gamma],
                                             tokens[d0:d0 + w.gamma], w.seed, r)
        return res.accepted_len

    def step():
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            return np.array(list(ex.map(one, range(n_req))))

    for _ in range(args.warmup):
        step()
    times, byts = [], []
    for _ in range(args.steps):
        s0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - s0)
        byts.append((2 * w.gamma + 1) * n_req * w.V * 2)  # algorithmic bytes, as our arm
    tot = sum(times)
    value = sum(byts) / tot / 1e9
    sample = (f"{n_req} of the 64 requests per step ({w.gamma} drafted positions each, "
              f"V={w.V}), threads over requests")
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": token_config(w, world),
            "impl": "reference",
            "positions_per_s": round(w.gamma * n_req * args.steps / tot, 2),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
