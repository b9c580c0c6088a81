"""Throughput of batched draft-token verification on GB300.

One step = one spec_verify_stochastic call on the headline workload (B=256 sequences,
gamma=8 drafts, V=128256, bf16 logits, T=0.6): temperature softmax of every target and
draft row, acceptance, first rejection, residual or bonus token, per-position NKL with
its delta=0.15 mask and the greedy decision, all from one read of the logits. The
metric is verified target rows per second (B*(gamma+1) rows per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank verifies its own batch (weak scaling, no collective on the
data path); rank 0 prints one JSON line. `--impl reference` times the fp64 CPU oracle
instead, on a bounded sample of the same workload."""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified rows/s & HBM GB/s vs GB300 peak (B=256, gamma=8, V=128256, bf16)"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def datasheet_gbs():
    """Nominal HBM3e bandwidth of a GB300: the memory clock (MEASURED_PEAKS.json
    mem_max_mhz, else 3996 MHz) x 2 transfers per clock x an 8192-bit bus."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["mem_max_mhz"])
    except Exception:
        mhz = 3996.0
    return mhz * 1e6 * 2 * 8192 / 8 / 1e9


PROFILE = os.path.join(ROOT, "profiles", "stochastic_call_B256_g8_V128256.md")


def kernel_sources_sha256() -> str:
    """Hash of the CUDA sources, the host planning header and the C header (the same recipe
    as the profile summary)."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "speculative_decoding_token_temp_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                   glob.glob(os.path.join(csrc, "*.h")))
    files.append(os.path.join(ROOT, "include", "spec_verify.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per call from the committed ncu summary, or None when the kernels have
    changed since it was taken (or it is missing)."""
    try:
        with open(PROFILE) as f:
            text = f.read()
        kv = {}
        for line in text.splitlines():
            line = line.strip()
            if ":" in line and line.split(":")[0] in ("sources_sha256", "traffic_bytes_per_call"):
                k, v = line.split(":", 1)
                kv[k] = v.strip()
        if kv.get("sources_sha256") != kernel_sources_sha256():
            return None
        return int(kv["traffic_bytes_per_call"])
    except Exception:
        return None


def algorithmic_bytes(w) -> dict:
    """Bytes the verification must read: every target and draft logit once, plus one
    (target, draft) row pair per sequence for the residual / bonus sample."""
    es = w.elem_bytes
    t = w.total_target * w.V * es
    d = w.total_draft * w.V * es
    resid = w.B * 2 * w.V * es
    small = w.total_draft * (4 + 4) + w.B * 4
    return {"stochastic": t + d + resid + small, "greedy": t + w.total_draft * 4, "nkl": w.total_draft * w.V * es * 2}


# ---------------------------------------------------------------- distributed plumbing

def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    from speculative_decoding_token_temp_gb300 import sharding
    return sharding.max_over_ranks(x, world, device)


def sum_over_ranks(x: float, world: int, device) -> float:
    from speculative_decoding_token_temp_gb300 import sharding
    return sharding.sum_over_ranks(x, world, device)


# ---------------------------------------------------------------- clocks

CLOCK_Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
           "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
           "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

def _to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _shifted(t, offset):
    """A copy of device tensor t that starts `offset` elements into its buffer (offset > 0
    puts the rows off the 16-byte grid: the library's phased path, every row at one
    offset)."""
    import torch
    if offset == 0:
        return t
    buf = torch.empty(t.numel() + offset, dtype=t.dtype, device=t.device)
    buf[offset:].copy_(t.reshape(-1))
    return buf[offset:].view(t.shape)


class StochasticCall:
    """Preallocated inputs/outputs for repeated spec_verify_stochastic calls (logits
    shifted by `offset` elements when offset > 0)."""

    def __init__(self, w, dev, host_inputs=False, offset=0, temperature_draft=None):
        import ctypes

        import torch

        from speculative_decoding_token_temp_gb300 import _lib
        self.w = w
        self.dev = dev
        self.lib = _lib.lib()
        B, V = w.B, w.V
        rows, tot = w.total_target, w.total_draft
        self.t = _shifted(_to_dev(w.target, dev), offset)
        self.d = _shifted(_to_dev(w.draft, dev), offset)
        self.tok = _to_dev(w.tokens, dev)
        self.ua = _to_dev(w.u_accept, dev)
        self.us = _to_dev(w.u_sample, dev)
        self.cu = None if w.dense else _to_dev(w.cu_draft, dev)
        z = lambda n, dt: torch.empty(n, dtype=dt, device=dev)  # noqa: E731
        self.n = z(B, torch.int32)
        self.out = z(rows, torch.int32)
        self.px, self.qx, self.al, self.nkl = (z(tot, torch.float32) for _ in range(4))
        self.mask = z(tot, torch.uint8)
        self.gn = z(B, torch.int32)
        self.gt = z(rows, torch.int32)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.g = _lib.SpecBatch(B, w.gamma_max if not w.dense else int(w.gammas[0]), V, tot,
                                ctypes.c_void_p(self.cu.data_ptr()) if self.cu is not None else None)
        nbytes = self.lib.spec_workspace_bytes(self.g, _lib.SPEC_BF16 if w.dtype == 'bf16' else _lib.SPEC_F32, _lib.SPEC_MODE_STOCHASTIC)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.dt = _lib.SPEC_BF16 if w.dtype == "bf16" else _lib.SPEC_F32
        self.host = None
        self.P = ctypes.c_void_p
        self.opts = None
        if temperature_draft is not None:  # spec_verify_stochastic_ex with the draft's own temperature
            self.opts = _lib.SpecOptions()
            self.opts.temperature_draft = float(temperature_draft)
        self.ins = [{"t": self.t, "d": self.d, "tok": self.tok, "ua": self.ua, "us": self.us}]
        if host_inputs:
            pin = lambda t: t.cpu().pin_memory()  # noqa: E731
            self.host = {"t": pin(self.t), "d": pin(self.d), "tok": pin(self.tok), "ua": pin(self.ua),
                         "us": pin(self.us)}
            self.host_out = {"n": torch.empty(B, dtype=torch.int32).pin_memory(),
                             "out": torch.empty(rows, dtype=torch.int32).pin_memory()}
            # end to end, double-buffered: the inputs of step i + 1 cross the link on a copy
            # stream while step i is verified from the other set of device buffers
            self.ins.append({"t": _shifted(torch.empty_like(self.t), offset),
                             "d": _shifted(torch.empty_like(self.d), offset),
                             "tok": torch.empty_like(self.tok), "ua": torch.empty_like(self.ua),
                             "us": torch.empty_like(self.us)})
            self.copy_stream = torch.cuda.Stream(dev)
            self.copied = [torch.cuda.Event(), torch.cuda.Event()]
            self.consumed = [torch.cuda.Event(), torch.cuda.Event()]
            self.e2e_i = 0

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.host.values())

    def d2h_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.host_out.values())

    def __call__(self, stream_handle, k=0):
        import ctypes
        P = self.P
        x = self.ins[k]
        args = (self.g, self.dt, P(x["t"].data_ptr()), P(x["d"].data_ptr()), P(x["tok"].data_ptr()), self.w.T,
                P(x["ua"].data_ptr()), P(x["us"].data_ptr()), P(self.n.data_ptr()), P(self.out.data_ptr()),
                P(self.px.data_ptr()), P(self.qx.data_ptr()), P(self.al.data_ptr()), P(self.nkl.data_ptr()),
                P(self.mask.data_ptr()), 0.15, P(self.gn.data_ptr()), P(self.gt.data_ptr()))
        tail = (P(self.status.data_ptr()), P(self.ws.data_ptr()), self.ws.numel(), P(stream_handle))
        if self.opts is None:
            code = self.lib.spec_verify_stochastic(*args, *tail)
        else:
            code = self.lib.spec_verify_stochastic_ex(*args, ctypes.byref(self.opts), *tail)
        if code != 0:
            raise RuntimeError(f"spec_verify_stochastic returned {code}")

    def e2e_step(self, stream):
        """One end-to-end step: this step's inputs copied from pinned host memory into buffer
        set k = step % 2 on the copy stream, once the call that last read set k (two steps
        back) is done; the call on `stream` once they have landed; its decisions copied back to
        pinned host memory on `stream`. One step's copies thus overlap the previous call."""
        import torch
        k = self.e2e_i % 2
        self.e2e_i += 1
        x = self.ins[k]
        cs = self.copy_stream
        cs.wait_event(self.consumed[k])  # a no-op before the event is first recorded
        with torch.cuda.stream(cs):
            for name in ("t", "d", "tok", "ua", "us"):
                x[name].copy_(self.host[name], non_blocking=True)
            self.copied[k].record(cs)
        stream.wait_event(self.copied[k])
        self(stream.cuda_stream, k)
        self.consumed[k].record(stream)
        self.host_out["n"].copy_(self.n, non_blocking=True)
        self.host_out["out"].copy_(self.out, non_blocking=True)


def time_loop(fn, steps, warmup, stream, world, dev):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    return a.elapsed_time(b) / 1e3


def time_e2e(call, steps, warmup, stream, world, dev):
    """Seconds for `steps` end-to-end steps (StochasticCall.e2e_step): events on `stream`
    bracket them, the copy stream starts after the first event, and the last step's
    read-back (after its call, after its copies) precedes the second."""
    import torch
    for _ in range(warmup):
        call.e2e_step(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    call.copy_stream.wait_stream(stream)
    for _ in range(steps):
        call.e2e_step(stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    return a.elapsed_time(b) / 1e3


def time_mode(fn, steps, warmup, dev):
    """Per-call device time of a secondary mode (single GPU, no barrier). When one call's
    host cost is comparable to its device time, a plain loop measures the host; so a
    bounded sleep kernel queued first holds the stream while the host enqueues the timed
    calls (at most 100, well inside the launch queue), and the events then bracket the
    calls running back to back on the device."""
    import torch
    s = torch.cuda.current_stream(dev)
    t0 = time.perf_counter()
    for _ in range(warmup):
        fn()
    host = (time.perf_counter() - t0) / max(warmup, 1)       # per call, enqueue included
    torch.cuda.synchronize(dev)
    steps = min(steps, 100)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(min(2e8, 2.5e9 * host * steps * 1.5)))   # GPU clock cycles (<= ~0.1 s)
    a.record(s)
    for _ in range(steps):
        fn()
    b.record(s)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / 1e3 / steps


def time_cold(fn, reps, warmup, dev):
    """Per-call device time with a cold L2: before every call a buffer of at least twice the
    L2 size is written and then a second one read, so the call finds none of its inputs in
    L2 and no dirty line of the flush is written back during it; CUDA events bracket the
    call alone on the launching stream. Returns (median, 10th, 90th percentile) seconds."""
    import torch
    s = torch.cuda.current_stream(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    nbytes = max(2 * l2, 256 << 20)
    wbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(reps):
        wbuf.zero_()
        rbuf.sum()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    del wbuf, rbuf
    times.sort()
    return times[len(times) // 2], times[len(times) // 10], times[(len(times) * 9) // 10]


def _oracle_worker(seed, seqs, gamma, V, dtype, T, agreement, barrier, q):
    """One process of the all-cores baseline: regenerate its sequences (untimed), wait for
    the others, then run the oracle on them and report (rows, seconds)."""
    import time as _t

    from oracle import oracle as O
    from speculative_decoding_token_temp_gb300 import synth
    data = [synth.sequence_data(seed, b, gamma, V, dtype, T, agreement) for b in seqs]
    barrier.wait()
    t0 = _t.perf_counter()
    rows = 0
    for t_st, d_st, tok, ua, us in data:
        O.verify_stochastic_sequence(O.widen(t_st, dtype), O.widen(d_st, dtype), tok, T, ua.astype("float64"),
                                     float(us))
        rows += len(tok) + 1
    q.put((rows, _t.perf_counter() - t0))


def cpu_baseline_all_cores(cfg, seed, B, nproc=None):
    """The oracle on every host core: one spawned process per core (the GPU is already in
    use, so no fork), each on its share of the B sequences; rows / slowest process."""
    import multiprocessing as mp
    nproc = nproc or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(nproc)
    q = ctx.Queue()
    shares = [list(range(r, B, nproc)) for r in range(nproc)]
    procs = [ctx.Process(target=_oracle_worker, args=(seed, shares[r], cfg.gamma, cfg.V, cfg.dtype, cfg.T[0],
                                                      cfg.agreement, barrier, q)) for r in range(nproc)]
    for pr in procs:
        pr.start()
    import queue as _queue
    res = []
    deadline = time.time() + 600
    while len(res) < nproc:
        try:
            res.append(q.get(timeout=2))
        except _queue.Empty:
            if any(pr.exitcode not in (None, 0) for pr in procs) or time.time() > deadline:
                for pr in procs:
                    if pr.is_alive():
                        pr.terminate()
                return None
    for pr in procs:
        pr.join(timeout=60)
    rows = sum(r for r, _ in res)
    slowest = max(t for _, t in res)
    return {"value": rows / slowest, "unit": "rows/s", "cores": nproc, "kind": "oracle",
            "sample": f"all {B} sequences ({rows} target rows) of the {cfg.name} workload, "
                      f"stochastic+NKL+greedy in fp64 numpy, {nproc} processes (one per host core), "
                      f"slowest {slowest:.2f} s"}


def cpu_baseline(w, budget_s=12.0):
    """The fp64 oracle as it stands on this host: stochastic + NKL + greedy per sequence,
    sequences taken in order until the time budget is spent."""
    from oracle import oracle as O
    t0 = time.perf_counter()
    rows = 0
    done = 0
    for b in range(w.B):
        O.verify_stochastic(w.target, w.draft, w.tokens, w.cu_draft, w.T, w.u_accept, w.u_sample, w.dtype,
                            seqs=[b])
        rows += int(w.gammas[b]) + 1
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": rows / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.B} sequences ({rows} target rows) of the B=256/gamma=8/V=128256 bf16 "
                      f"workload, stochastic+NKL+greedy in fp64 numpy, single thread, {el:.1f} s"}


def run_ours(args):
    import torch

    import __graft_entry__
    from speculative_decoding_token_temp_gb300 import api, synth

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    __graft_entry__.build()
    cfg = synth.HEADLINE
    from speculative_decoding_token_temp_gb300 import sharding
    w = cfg.make(seed=sharding.rank_seed(cfg.seed, rank), B=args.batch, V=args.vocab)
    call = StochasticCall(w, dev, host_inputs=True, offset=args.offset, temperature_draft=args.temperature_draft)
    secondary = args.offset != 0 or args.temperature_draft is not None
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    step = lambda: call(sh)  # noqa: E731

    clocks = ClockSampler(local)
    time.sleep(0.3)
    el = time_loop(step, args.steps, args.warmup, stream, world, dev)
    ck = clocks.stop()
    el = max_over_ranks(el, world, dev)
    status = int(call.status.item())
    rows_step = w.total_target
    total_rows = sum_over_ranks(rows_step * args.steps, world, dev)
    value = total_rows / el
    ms = el / args.steps * 1e3

    hbm, peak_kind = peaks()
    ab = algorithmic_bytes(w)
    achieved = ab["stochastic"] / (ms / 1e3) / 1e9

    # end to end: host buffers, H2D of every input and D2H of the decisions inside the timed region
    ref_n, ref_out = call.n.cpu(), call.out.cpu()  # the device-resident run's decisions, same inputs
    e2e_steps = max(3, min(20, args.steps))
    e2e_el = time_e2e(call, e2e_steps, 2, stream, world, dev)
    e2e_same = bool(torch.equal(call.host_out["n"], ref_n) and torch.equal(call.host_out["out"], ref_out))
    e2e_el = max_over_ranks(e2e_el, world, dev)
    e2e_val = sum_over_ranks(rows_step * e2e_steps, world, dev) / e2e_el

    modes = {}
    if rank == 0 and not args.no_modes and w.V == cfg.V and args.temperature_draft is None:
        # the standalone calls, same inputs (the workload's own vocabulary only)
        res = {}
        g_out = {}
        gfn = lambda: api.spec_verify_greedy(call.t, call.tok, gamma=8, out=g_out)  # noqa: E731
        t_g = time_mode(gfn, 200, 10, dev)
        modes["greedy_B256_g8_V128256"] = {"us_per_call": t_g * 1e6,
                                           "GBps": ab["greedy"] / t_g / 1e9, "rows_per_s": rows_step / t_g}
        n_out = {}
        nfn = lambda: api.spec_nkl(call.t, call.d, w.T, gamma=8, out=n_out)  # noqa: E731
        t_n = time_mode(nfn, 200, 10, dev)
        modes["nkl_B256_g8_V128256"] = {"us_per_call": t_n * 1e6, "GBps": ab["nkl"] / t_n / 1e9}
        # policy variants (spec_options) on the same inputs
        st = api.new_accept_stats(dev)
        pos = torch.arange(1, w.B + 1, dtype=torch.int32, device=dev) * 37
        gam = int(w.gammas[0])
        x_out = {}
        xfn = lambda: api.spec_verify_stochastic_ex(call.t, call.d, call.tok, w.T, call.ua, call.us,  # noqa: E731
                                                    gamma=gam, out=x_out, temperature_draft=0.4)
        t_x = time_mode(xfn, 200, 10, dev)
        modes["stochastic_draft_T0.4_B256_g8_V128256"] = {
            "us_per_call": t_x * 1e6, "GBps": ab["stochastic"] / t_x / 1e9,
            "frac_of_peak": ab["stochastic"] / t_x / 1e9 / hbm,
            "note": "target T 0.6, drafts at T_d 0.4, with the NKL outputs: the draft rows are summed at "
                    "both temperatures"}
        xn_out = {}
        xnfn = lambda: api.spec_verify_stochastic_ex(call.t, call.d, call.tok, w.T, call.ua, call.us,  # noqa: E731
                                                     gamma=gam, out=xn_out, temperature_draft=0.4, want_nkl=False)
        t_xn = time_mode(xnfn, 200, 10, dev)
        modes["stochastic_draft_T0.4_no_nkl_B256_g8_V128256"] = {
            "us_per_call": t_xn * 1e6, "GBps": ab["stochastic"] / t_xn / 1e9,
            "frac_of_peak": ab["stochastic"] / t_xn / 1e9 / hbm,
            "note": "the same without the NKL outputs: the draft rows at T_d only (single-scale tiles)"}
        a_out = {}
        afn = lambda: api.spec_verify_stochastic_ex(call.t, call.d, call.tok, w.T, call.ua, call.us,  # noqa: E731
                                                    gamma=gam, out=a_out, position=pos, min_block_len=3,
                                                    stats=st, stats_bucket=1)
        t_a = time_mode(afn, 200, 10, dev)
        modes["stochastic_position_block_stats_B256_g8_V128256"] = {
            "us_per_call": t_a * 1e6, "GBps": ab["stochastic"] / t_a / 1e9,
            "frac_of_peak": ab["stochastic"] / t_a / 1e9 / hbm}
        gp_out = {}
        gpfn = lambda: api.spec_verify_greedy_ex(call.t, call.tok, gamma=gam, out=gp_out,  # noqa: E731
                                                 min_block_len=3, stats=st, stats_bucket=2)
        t_gp = time_mode(gpfn, 200, 10, dev)
        modes["greedy_block_stats_B256_g8_V128256"] = {"us_per_call": t_gp * 1e6, "GBps": ab["greedy"] / t_gp / 1e9}
        # multi-draft: 64 groups of 3 candidates with the headline's gamma, V and dtype
        wm = synth.make_multi(64, 3, gam, w.V, w.dtype, w.T, seed=5)
        tm, dm, km = _to_dev(wm.target, dev), _to_dev(wm.draft, dev), _to_dev(wm.tokens, dev)
        uam, usm = _to_dev(wm.u_accept, dev), _to_dev(wm.u_sample, dev)
        m_out = {}
        mfn = lambda: api.spec_verify_multi(tm, dm, km, 3, wm.T, stochastic=True, u_accept=uam,  # noqa: E731
                                            u_sample=usm, out=m_out)
        t_m = time_mode(mfn, 100, 5, dev)
        eb = 2 if w.dtype == synth.BF16 else 4
        mb_min = (wm.target.size + wm.draft.size + 2 * wm.B * wm.V) * eb
        modes["multi_draft_G64_K3_g8_V128256"] = {
            "us_per_call": t_m * 1e6, "GBps": mb_min / t_m / 1e9, "frac_of_peak": mb_min / t_m / 1e9 / hbm,
            "note": "algorithmic bytes: every logit once + one row pair per candidate; the fused K-way tiles "
                    "read every logit once (rows off the 16-byte grid take the two-pass form, which reads "
                    f"the draft rows a second time: +{wm.draft.size * eb / 1e6:.0f} MB)"}
        del tm, dm, km, uam, usm, m_out
        sm_out = torch.empty(6, dtype=torch.float64, device=dev)
        t_sm = time_mode(lambda: api.spec_accept_summary(st, 2, 64, out=sm_out), 200, 10, dev)
        modes["accept_summary_64_slots"] = {"us_per_call": t_sm * 1e6,
                                            "note": "one 64-thread block; the figure includes the host's enqueue rate"}
        if args.offset == 0:
            # the same call with the logits one element off the 16-byte grid: the phased path
            ts, ds = _shifted(call.t, 1), _shifted(call.d, 1)
            s_out = {}
            sfn = lambda: api.spec_verify_stochastic(ts, ds, call.tok, w.T, call.ua, call.us,  # noqa: E731
                                                     gamma=gam, out=s_out)
            t_s = time_mode(sfn, 200, 10, dev)
            sg_out = {}
            t_sg = time_mode(lambda: api.spec_verify_greedy(ts, call.tok, gamma=gam, out=sg_out), 200, 10, dev)
            modes["stochastic_offset1_B256_g8_V128256"] = {
                "us_per_call": t_s * 1e6, "GBps": ab["stochastic"] / t_s / 1e9,
                "frac_of_peak": ab["stochastic"] / t_s / 1e9 / hbm, "greedy_us_per_call": t_sg * 1e6,
                "note": "logits one element off the 16-byte grid (both rows of a pair at one offset): the "
                        "phased tiles stream the whole aligned blocks with the offset applied to the "
                        "indices, the partial blocks at the chunks' ends folded by the row merge "
                        "(stochastic) or the tiles' last threads (greedy)"}
            del ts, ds, s_out, sg_out
        del res
        tw = synth.TREE.make()
        tt = _to_dev(tw.target, dev)
        tn = _to_dev(tw.node_tokens, dev)
        t_out = {}
        tfn = lambda: api.spec_verify_tree(tt, tn, list(tw.parent), out=t_out)  # noqa: E731
        t_t = time_mode(tfn, 500, 10, dev)
        tbytes = tw.target.nbytes
        modes["tree_B32_N12_V128256"] = {"us_per_call": t_t * 1e6, "GBps": tbytes / t_t / 1e9,
                                         "rows_per_s": tw.B * (tw.N + 1) / t_t,
                                         "note": "back-to-back calls: the 107 MB of rows stay mostly in L2"}
        tc, tc10, tc90 = time_cold(tfn, 60, 5, dev)
        modes["tree_B32_N12_V128256_cold_L2"] = {
            "us_per_call": tc * 1e6, "us_p10": tc10 * 1e6, "us_p90": tc90 * 1e6, "GBps": tbytes / tc / 1e9,
            "frac_of_peak": tbytes / tc / 1e9 / hbm,
            "note": "median of 60 calls, each after L2 is flushed (a 2x-L2 buffer written, another read)"}
        del tt, tn
        w1 = synth.MID.make(T=0.6)
        c1 = StochasticCall(w1, dev)
        t_1 = time_mode(lambda: c1(sh), 500, 10, dev)
        b1 = algorithmic_bytes(w1)["stochastic"]
        modes["stochastic_B64_g5_V32000_warm_L2"] = {"us_per_call": t_1 * 1e6, "GBps": b1 / t_1 / 1e9,
                                                     "rows_per_s": w1.total_target / t_1,
                                                     "note": "53 MB of inputs fit in L2: warm-cache figure"}
        c1c, c1c10, c1c90 = time_cold(lambda: c1(sh), 60, 5, dev)
        modes["stochastic_B64_g5_V32000_cold_L2"] = {
            "us_per_call": c1c * 1e6, "us_p10": c1c10 * 1e6, "us_p90": c1c90 * 1e6, "GBps": b1 / c1c / 1e9,
            "frac_of_peak": b1 / c1c / 1e9 / hbm, "rows_per_s": w1.total_target / c1c,
            "note": "median of 60 calls, each after L2 is flushed (a 2x-L2 buffer written, another read)"}
        del c1
        # a vocabulary whose bf16 row is not a whole number of 16-byte blocks: every row has
        # its own offset within the grid, and the rows of a pair differ (shifted pair tiles)
        w5 = synth.make_stochastic(256, 50257, synth.BF16, 0.6, seed=7, gamma=8, name="B256_g8_V50257_bf16")
        c5 = StochasticCall(w5, dev)
        t_5 = time_mode(lambda: c5(sh), 200, 10, dev)
        b5 = algorithmic_bytes(w5)["stochastic"]
        g5_out = {}
        t_5g = time_mode(lambda: api.spec_verify_greedy(c5.t, c5.tok, gamma=8, out=g5_out), 200, 10, dev)
        modes["stochastic_B256_g8_V50257"] = {
            "us_per_call": t_5 * 1e6, "GBps": b5 / t_5 / 1e9, "frac_of_peak": b5 / t_5 / 1e9 / hbm,
            "rows_per_s": w5.total_target / t_5, "greedy_us_per_call": t_5g * 1e6,
            "greedy_frac_of_peak": algorithmic_bytes(w5)["greedy"] / t_5g / 1e9 / hbm,
            "note": "rows of 50257 bf16 (not a whole number of 16-byte blocks): the pair tiles shift the draft "
                    "rows' vectors to the target rows' offset, and the sampler reads them the same way"}
        del c5, w5, g5_out
        if not args.skip_ragged:
            w4 = synth.RAGGED.make()
            c4 = StochasticCall(w4, dev)
            t_4 = time_mode(lambda: c4(sh), 100, 5, dev)
            b4 = algorithmic_bytes(w4)["stochastic"]
            modes["stochastic_ragged_B512_V152064"] = {"us_per_call": t_4 * 1e6, "GBps": b4 / t_4 / 1e9,
                                                       "rows_per_s": w4.total_target / t_4,
                                                       "frac_of_peak": b4 / t_4 / 1e9 / hbm}
            del c4

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu:
        one = cpu_baseline(w)
        allc = cpu_baseline_all_cores(cfg, cfg.seed, w.B) if w.dense and w.B == cfg.B and w.V == cfg.V else None
        if allc is not None:
            allc["single_thread"] = one
        cpu = allc if allc is not None else one
    out = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"B{w.B}_g8_V{w.V}_bf16: stochastic verify + NKL(delta=0.15) + greedy, one call"
                               + (f" (logits {args.offset} element(s) off the 16-byte grid: phased path)"
                                  if args.offset else "")
                               + (f" (draft temperature {args.temperature_draft}: both draft scales)"
                                  if args.temperature_draft is not None else ""),
                   "B": w.B, "gamma": 8, "V": w.V, "T": w.T, "seed": cfg.seed, "rows_per_step": rows_step,
                   "l2": f"inputs {(w.target.nbytes + w.draft.nbytes) / 1e6:.0f} MB per step, larger than the "
                         "129 MB L2; no flush",
                   "parallelism": f"{world} independent shard(s), no collective"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": profiled_traffic() if w.B == 256 and w.V == cfg.V and not secondary else None,
                     "kernel": "spec_verify_stochastic call (prologue_kernel + rows_kernel + sample2_kernel)",
                     "algorithmic_bytes": ab["stochastic"], "peak_source": peak_kind,
                     "peak_datasheet": datasheet_gbs(), "frac_datasheet": achieved / datasheet_gbs(),
                     "note": f"achieved = algorithmic bytes / call time (CUDA events); frac uses peak = the {peak_kind} "
                             "MEASURED_PEAKS.json hbm_gbs (a copy: it reads and writes, the call only reads); "
                             "frac_datasheet uses the memory clock x 2 x 8192-bit HBM3e bus; traffic = DRAM "
                             "bytes per call copied from the committed ncu summary (profiles/"
                             "stochastic_call_B256_g8_V128256.md) while the CUDA sources hash to the profiled "
                             "ones, else null"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "rows/s", "h2d_bytes_per_step": call.h2d_bytes(),
                "d2h_bytes_per_step": call.d2h_bytes(), "decisions_match_device_run": e2e_same},
        "gpu_launches": 3 * args.steps,
        "clocks": ck,
        "device_status": status,
        "modes": modes,
    }
    print(json.dumps(out))


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    """The fp64 oracle on the host cores, on the same workload. Each step verifies a
    bounded sample: m whole sequences, or, when K+W steps of one sequence each would
    not finish in about two minutes, the first k positions of a sequence (a sub-sequence
    whose last target row serves as its bonus row), k and m sized from one calibration
    sequence."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as O
    from speculative_decoding_token_temp_gb300 import synth
    cfg = synth.HEADLINE
    g = cfg.gamma
    budget = 120.0
    cal = synth.make_stochastic(1, cfg.V, cfg.dtype, cfg.T[0], cfg.seed + 77, gamma=g)
    t0 = time.perf_counter()
    O.verify_stochastic(cal.target, cal.draft, cal.tokens, cal.cu_draft, cal.T, cal.u_accept, cal.u_sample,
                        cal.dtype)
    t_seq = time.perf_counter() - t0
    per_step = budget / (args.steps + args.warmup)
    m = int(max(1, min(3, per_step // t_seq)))
    k = g if per_step >= t_seq else int(max(1, min(g, (per_step / t_seq) * (g + 1) - 1)))
    nseq = m * (args.steps + args.warmup) if k == g else (args.steps + args.warmup)
    pool = min(nseq, 64)
    w = synth.make_stochastic(pool, cfg.V, cfg.dtype, cfg.T[0], cfg.seed, gamma=g)
    widen = lambda a: O.widen(a, w.dtype)  # noqa: E731
    step_i = 0

    def step():
        nonlocal step_i
        if k == g:
            seqs = [(step_i * m + j) % pool for j in range(m)]
            O.verify_stochastic(w.target, w.draft, w.tokens, w.cu_draft, w.T, w.u_accept, w.u_sample, w.dtype,
                                seqs=seqs)
        else:
            b = step_i % pool
            t_rows, d_rows, tok, ua, us = w.sequence(b)
            O.verify_stochastic_sequence(widen(t_rows[:k + 1]), widen(d_rows[:k]), tok[:k], w.T,
                                         ua[:k].astype(np.float64), us)
        step_i += 1

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    rows_per_step = m * (g + 1) if k == g else k + 1
    val = rows_per_step * args.steps / el
    sample = (f"{m} whole sequence(s) per step" if k == g else f"the first {k} of {g} positions of one sequence "
              f"per step (+ its next target row as bonus row)")
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": "rows/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "B256_g8_V128256_bf16: stochastic verify + NKL(delta=0.15) + greedy",
                      "B": cfg.B, "gamma": g, "V": cfg.V, "T": cfg.T[0], "seed": cfg.seed,
                      "sample_per_step": sample},
           "cpu_baseline": {"value": val, "unit": "rows/s", "cores": 1, "kind": "oracle",
                            "sample": sample + f" ({rows_per_step} target rows), fp64 numpy, single thread"},
           "e2e": {"value": val, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-modes", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--skip-ragged", action="store_true")
    ap.add_argument("--offset", type=int, default=0, metavar="N",
                    help="shift the timed call's logits by N elements (N not a multiple of 8: the phased path)")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences per step (default: the workload's 256); smaller slices serve profiling")
    ap.add_argument("--vocab", type=int, default=None, metavar="V",
                    help="vocabulary of the timed call (default: the workload's 128256); a secondary line, e.g. "
                         "V=50257, whose rows are not whole 16-byte blocks (the shifted path), for profiling")
    ap.add_argument("--temperature-draft", type=float, default=None, metavar="T_D",
                    help="time the call with the drafts at their own temperature T_D (spec_verify_stochastic_ex, "
                         "NKL outputs kept: the tiles sum the draft row at both scales); a secondary line, for "
                         "profiling")
    ap.add_argument("--tree", action="store_true",
                    help="time only the tree call (B=32, 12 nodes, V=128256, bf16): back-to-back and with L2 flushed "
                         "before every call; a secondary line for profiling, not the headline metric")
    ap.add_argument("--multi", type=int, default=None, metavar="G",
                    help="time only the multi-draft call on G groups of 3 candidates (gamma 8, V 128256, bf16): "
                         "a secondary line for profiling, not the headline metric")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.tree:
        run_tree_only(args)
    elif args.multi is not None:
        run_multi_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


def run_tree_only(args):
    """spec_verify_tree on the 12-node tree workload (B=32, V=128256, bf16): per-call device
    time back to back (the rows stay mostly in L2) and cold (L2 flushed before every call),
    with GB/s of the target rows."""
    import torch

    import __graft_entry__
    from speculative_decoding_token_temp_gb300 import api, synth
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    tw = synth.TREE.make()
    tt, tn = _to_dev(tw.target, dev), _to_dev(tw.node_tokens, dev)
    out = {}
    fn = lambda: api.spec_verify_tree(tt, tn, list(tw.parent), out=out)  # noqa: E731
    warm = time_mode(fn, args.steps, args.warmup, dev)
    cold, c10, c90 = time_cold(fn, max(args.steps, 10), args.warmup, dev)
    hbm, _ = peaks()
    print(json.dumps({"metric": "tree_us_per_call", "value": cold * 1e6, "unit": "us", "warm_us": warm * 1e6,
                      "cold_p10_us": c10 * 1e6, "cold_p90_us": c90 * 1e6,
                      "cold_frac_of_peak": tw.target.nbytes / cold / 1e9 / hbm,
                      "status": int(out["device_status"][0]),
                      "config": {"workload": "tree B=32 N=12 V=128256 bf16"}}))


def run_multi_only(args):
    """spec_verify_multi (stochastic) on make_multi(G, 3, 8, 128256, bf16): per-call device
    time and GB/s of the minimal bytes (every logit once + one row pair per candidate)."""
    import torch

    import __graft_entry__
    from speculative_decoding_token_temp_gb300 import api, synth
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    w = synth.make_multi(args.multi, 3, 8, 128256, synth.BF16, 0.6, seed=5)
    t, d, k = _to_dev(w.target, dev), _to_dev(w.draft, dev), _to_dev(w.tokens, dev)
    ua, us = _to_dev(w.u_accept, dev), _to_dev(w.u_sample, dev)
    out = {}
    fn = lambda: api.spec_verify_multi(t, d, k, 3, w.T, stochastic=True, u_accept=ua, u_sample=us,  # noqa: E731
                                       out=out)
    sec = time_mode(fn, args.steps, args.warmup, dev)
    minimal = (w.target.size + w.draft.size + 2 * w.B * w.V) * 2
    hbm, _ = peaks()
    print(json.dumps({"metric": "multi_draft_us_per_call", "value": sec * 1e6, "unit": "us",
                      "GBps": minimal / sec / 1e9, "frac_of_peak": minimal / sec / 1e9 / hbm,
                      "status": int(out["device_status"][0]),
                      "config": {"workload": f"multi-draft G={args.multi} K=3 gamma=8 V=128256 bf16"}}))


if __name__ == "__main__":
    main()
