#!/usr/bin/env python
"""Benchmark of the W4A16 verify hot path on GB300.

One step is one pass over every configuration the metric spans, T = 1..32,
with the shapes of a 27B-class decoder (fused QKV 5120->10240, fused gate+up
5120->34816, down 17408->5120, int4 lm_head 248,320 x 5,120, a 40,960-id
restricted draft head):

  leg              calls (in order)
  decode_T1        the three GEMMs at T = 1
  mtp_T4           the three GEMMs at T = 4, then the lm_head verify (3 drafts)
  dflash2_T8       the three GEMMs at T = 8, then the lm_head verify (7 drafts)
  dflash2_4x8_T32  the three GEMMs at T = 32, then one lm_head pass verifying
                   four streams of 1 + 7 rows
  restricted_T1    the restricted head over 40,960 mapped rows, T = 1
  restricted_T4    the restricted head, T = 4 (3 drafts)

Every leg has its own weights, so the step streams 2.85 GB (far more than the
129 MB L2) and every call reads its weights from HBM.  The metric is
algorithmic HBM bytes per second (weights + scales read once, activations,
id list and drafts read, outputs written).  Inputs are seeded synthetic data.

Usage: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
                       [--breakdown] [--ncu-case ...]
One JSON line on stdout (rank 0).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "W4A16 skinny-GEMM + lm_head verify HBM GB/s (frac of 8 TB/s), T=1..32"
NOMINAL_HBM_GBS = 8000.0
WORKLOAD = "sweep_T1_T4_T8_T32_restricted"

# (leg name, config index, seed, T, GEMMs?, head: (n_draft, n_streams, n_map) or None)
LEGS = (
    ("decode_T1", 1, 1, 1, True, None),
    ("mtp_T4", 2, 2, 4, True, (3, 1, 0)),
    ("dflash2_T8", 3, 3, 8, True, (7, 1, 0)),
    ("dflash2_4x8_T32", 3, 33, 32, True, (7, 4, 0)),
    ("restricted_T1", 4, 4, 1, False, (0, 1, gen.DRAFT_VOCAB)),
    ("restricted_T4", 4, 44, 4, False, (3, 1, gen.DRAFT_VOCAB)),
)


def workload_config():
    """The workload, as both arms print it."""
    return {"workload": WORKLOAD,
            "legs": [{"leg": n, "config": c, "T": T,
                      "gemms": [list(s) for s in gen.GEMM_SHAPES] if g else [],
                      "head": None if h is None else {"V": gen.VOCAB, "K": gen.HIDDEN, "n_draft": h[0],
                                                      "n_streams": h[1], "n_map": h[2]}}
                     for n, c, _, T, g, h in LEGS],
            "bytes_per_step": step_bytes(),
            "l2": "inputs larger than L2 (2.85 GB streamed per step, every leg with its own weights)",
            "seeds": {n: s for n, _, s, _, _, _ in LEGS}}


def head_bytes(T, head):
    n_draft, S, n_map = head
    return gen.lmhead_bytes(gen.VOCAB, gen.HIDDEN, T, n_map=n_map, n_streams=S, n_draft=n_draft)


def leg_bytes(leg):
    _, _, _, T, g, h = leg
    b = sum(gen.gemm_bytes(T, K, N) for _, K, N in gen.GEMM_SHAPES) if g else 0
    return b + (head_bytes(T, h) if h is not None else 0)


def step_bytes():
    return sum(leg_bytes(leg) for leg in LEGS)


def kernels_per_call(T):
    """Kernel launches of one library call: the stream kernel, plus the
    activation conversion kernel when the call has more than one token tile
    (T > 8)."""
    return 2 if T > 8 else 1


def kernel_of(c):
    """The kernel the library dispatches a bench call to (its rule, for the
    shapes here): tcgen05 for 17..32 tokens, the 512-row kernel for a full-
    vocabulary head of 9..16 tokens, the stream kernel otherwise."""
    if c["T"] > 16:
        return "w4a16_tc_kernel"
    if c["T"] > 8 and c["kind"] == "head" and c.get("vm") is None:
        return "w4a16_wide_kernel"
    return "w4a16_stream_kernel"


# ----------------------------------------------------------------------------
# helpers


def reduce_max(dist, x, device=None):
    """The largest x over all ranks (a whole-job time is the slowest rank's);
    x itself when there is no process group.  NCCL reduces a device tensor,
    gloo a host one."""
    if dist is None:
        return float(x)
    import torch
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, bytes_per_step, steps, ms):
    """Whole-job throughput (weak scaling: every rank streams one step's
    bytes per step) over the slowest rank's time `ms` for `steps` steps."""
    return world * bytes_per_step * steps / (ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = {
    "w4a16_stream_kernel": ("w4a16_stream.cuh", "sv_ptx.cuh"),
    "w4a16_wide_kernel": ("w4a16_stream.cuh", "w4a16_wide.cuh", "sv_ptx.cuh"),
    "w4a16_tc_kernel": ("w4a16_stream.cuh", "w4a16_wide.cuh", "w4a16_tc.cuh", "sv_ptx.cuh"),
}


def code_only(src):
    """C++ source without its comments and with runs of whitespace made one
    space: what the compiler sees of it."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_digest(kernel="w4a16_stream_kernel", read=None):
    """Digest of the device code a kernel is compiled from (its sources
    without comments); ncu counters recorded for another digest describe a
    different kernel and are not reported.  `read(name)` gives a source's
    text (default: the working tree's file)."""
    csrc = os.path.join(ROOT, "speculative_verify_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        h.update(code_only(read(name)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(call, kernel):
    """DRAM bytes per launch of the bench call `call` (run by `kernel`) from
    the committed ncu summary, if it was taken on the kernel's current
    sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = kernel_source_digest(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == call and parts[1] == digest:
                return int(parts[2])
    return None


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model Name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU through
    NVML (read-only queries) every few milliseconds on a host thread."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, device, period_s=0.002):
        self.samples = []
        self.period = period_s
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            prop = torch.cuda.get_device_properties(device)
            bus = b"%08x:%02x:%02x.0" % (prop.pci_domain_id, prop.pci_bus_id, prop.pci_device_id)
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.nv, self.h = nv, h
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                r = 0
                if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                    r = int(rs.value)
                self.samples.append((time.perf_counter(), int(clk.value), r))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self, t0=None, t1=None):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable"}
        sel = [s for s in self.samples if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        window = "timed region"
        if not sel:          # region shorter than the sampling period: nearest samples
            mid = (t0 + t1) / 2 if t0 is not None else self.samples[-1][0]
            sel = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            window = "nearest samples to the timed region"
        mhz = float(np.median([s[1] for s in sel]))
        bits = 0
        for s in sel:
            bits |= s[2]
        reasons = [name for bit, name in self.REASONS.items() if bits & bit]
        return {"sm_mhz": mhz, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sel), "source": "nvml, " + window}


# ----------------------------------------------------------------------------
# host inputs (shared by the GPU arm and the oracle timing)


def host_leg(leg):
    """Seeded host inputs of one leg: per GEMM (x, Wq, scales); for the head
    (x, Wq, scales, drafts [S][n_draft], vocab_map or None)."""
    name, _, seed, T, g, h = leg
    rng = np.random.default_rng(seed)
    out = {"gemms": [], "head": None}
    if g:
        for label, K, N in gen.GEMM_SHAPES:
            Wq, sc = gen.weights(rng, N, K)
            out["gemms"].append((label, K, N, gen.activations(rng, T, K), Wq, sc))
    if h is not None:
        n_draft, S, n_map = h
        V, K = gen.VOCAB, gen.HIDDEN
        Wq, sc = gen.weights(rng, V, K)
        x = gen.activations(rng, T, K)
        vm = gen.vocab_map(rng, V, n_map) if n_map else None
        pool = vm if vm is not None else None
        if pool is None:
            drafts = rng.integers(0, V, size=(S, n_draft)).astype(np.int32)
        else:
            drafts = pool[rng.integers(0, pool.size, size=(S, n_draft))].astype(np.int32)
        out["head"] = (x, Wq, sc, drafts, vm)
    return out


# ----------------------------------------------------------------------------
# device workload


class Workload:
    """Device-resident inputs of the sweep step.  The per-call inputs of a
    step (every call's activations and drafts) are views of one device
    arena, and the verify results (accept_len, next_token of every verify
    stream) of one int32 array, so the end-to-end leg moves them with one
    copy each way."""

    def __init__(self, torch, device):
        dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)
        self.legs = []
        hosts = [host_leg(leg) for leg in LEGS]
        # arena: activations of every call, then drafts (16-byte aligned pieces)
        pieces = []
        for leg, hl in zip(LEGS, hosts):
            for (_, K, N, x, _, _) in hl["gemms"]:
                pieces.append(x.view(np.uint8).reshape(-1))
            if hl["head"] is not None:
                pieces.append(hl["head"][0].view(np.uint8).reshape(-1))
                pieces.append(hl["head"][3].view(np.uint8).reshape(-1))
        offs, o = [], 0
        for pc in pieces:
            offs.append(o)
            o += (pc.size + 15) // 16 * 16
        arena_host = np.zeros(o, np.uint8)
        for pc, off in zip(pieces, offs):
            arena_host[off:off + pc.size] = pc
        self.arena = torch.from_numpy(arena_host).to(device)
        n_out = sum(2 * h[1] for *_, h in LEGS if h is not None)
        self.out = torch.zeros(n_out, dtype=torch.int32, device=device)
        pi, oi = 0, 0

        def view(i, dt, shape):
            nb = pieces[i].size
            return self.arena[offs[i]:offs[i] + nb].view(dt).view(shape)

        for leg, hl in zip(LEGS, hosts):
            name, cfg, _, T, _, h = leg
            calls = []
            for (label, K, N, x, Wq, sc) in hl["gemms"]:
                xd = view(pi, torch.int16, (T, K))
                pi += 1
                calls.append(dict(kind="gemm", label="gemm_%s_T%d" % (label, T), T=T, K=K, N=N, x=xd,
                                  Wq=dev(Wq, np.int32), sc=dev(sc, np.int16),
                                  y=torch.empty((T, N), dtype=torch.bfloat16, device=device),
                                  bytes=gen.gemm_bytes(T, K, N), wbytes=N * K // 2 + N * K // 64))
            if h is not None:
                n_draft, S, n_map = h
                x, Wq, sc, drafts, vm = hl["head"]
                xd = view(pi, torch.int16, (T, gen.HIDDEN))
                dd = view(pi + 1, torch.int32, (S, n_draft))
                pi += 2
                acc = self.out[oi:oi + S]
                nxt = self.out[oi + S:oi + 2 * S]
                oi += 2 * S
                label = ("lmhead_verify_restricted_T%d" % T if n_map
                         else "lmhead_verify_T%d" % T if S == 1 else "lmhead_verify_%dx%d_T%d" % (S, n_draft + 1, T))
                calls.append(dict(kind="head", label=label, T=T, S=S, n_draft=n_draft, x=xd,
                                  Wq=dev(Wq, np.int32), sc=dev(sc, np.int16), drafts=dd,
                                  vm=None if vm is None else dev(vm, np.int32), acc=acc, nxt=nxt,
                                  bytes=head_bytes(T, h),
                                  wbytes=(n_map or gen.VOCAB) * (gen.HIDDEN // 2 + gen.HIDDEN // 64)))
            self.legs.append(dict(name=name, config=cfg, T=T, calls=calls, bytes=leg_bytes(leg)))
        self.bytes_per_step = sum(l["bytes"] for l in self.legs)
        self.launches_per_step = sum(kernels_per_call(c["T"]) for l in self.legs for c in l["calls"])
        self.host = hosts

    @staticmethod
    def call(sv, c, stream):
        if c["kind"] == "gemm":
            sv.w4a16_gemm(c["x"], c["Wq"], c["sc"], y=c["y"], stream=stream)
        elif c["vm"] is None:
            sv.lmhead_verify_batched(c["x"], c["Wq"], c["sc"], c["drafts"],
                                     accept_len=c["acc"], next_token=c["nxt"], stream=stream)
        else:
            # the draft vocabulary is model data: no kernel of the step writes it
            sv.lmhead_verify_ex(c["x"], c["Wq"], c["sc"], c["drafts"], vocab_map=c["vm"], flags=sv.MAP_STATIC,
                                accept_len=c["acc"], next_token=c["nxt"], stream=stream)

    def calls(self):
        return [c for l in self.legs for c in l["calls"]]

    def step(self, sv, stream):
        for c in self.calls():
            self.call(sv, c, stream)

    def capture(self, torch, sv, groups, prologue=None, epilogue=None):
        """One CUDA graph per group of calls (programmatic dependent launch
        between the kernels inside a graph); prologue/epilogue (optional)
        are captured before the first and after the last group's calls."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(side):
            for i, grp in enumerate(groups):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    if prologue is not None and i == 0:
                        prologue()
                    for c in grp:
                        self.call(sv, c, side)
                    if epilogue is not None and i == len(groups) - 1:
                        epilogue()
                graphs.append(g)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        return graphs


# ----------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)


def oracle_sample_step(oracle, hosts, rows_frac):
    """Run the oracle on a bounded sample of one sweep step: the first
    rows_frac of every GEMM's output rows and of every head's scored rows
    (for a restricted head, of its vocab_map), with the same x; the verify
    itself on the sampled logits.  Returns (algorithmic bytes, seconds)."""
    t0 = time.perf_counter()
    nbytes = 0
    for leg, hl in zip(LEGS, hosts):
        _, _, _, T, _, h = leg
        for (label, K, N, x, Wq, sc) in hl["gemms"]:
            n = max(1, int(N * rows_frac))
            oracle.w4a16_gemm(x, Wq[:n], sc[:n], T, K, n)
            nbytes += gen.gemm_bytes(T, K, n)
        if h is not None:
            n_draft, S, n_map = h
            x, Wq, sc, drafts, vm = hl["head"]
            V, K = Wq.shape[0], Wq.shape[1] * 8
            if vm is None:
                n = max(1, int(V * rows_frac))
                lg = oracle.lmhead_logits(x, Wq[:n], sc[:n], K, T, n)
                a, _, _ = oracle.argmax(lg)
                nbytes += gen.lmhead_bytes(n, K, T, n_streams=S, n_draft=n_draft)
            else:
                n = max(1, int(vm.size * rows_frac))
                lg = oracle.lmhead_logits(x, Wq, sc, K, T, V, rows=vm[:n])
                a, _, _ = oracle.argmax(lg, ids=vm[:n])
                nbytes += gen.lmhead_bytes(V, K, T, n_map=n, n_streams=S, n_draft=n_draft)
            for s in range(S):
                oracle.verify(a[s * (n_draft + 1):(s + 1) * (n_draft + 1)], drafts[s])
    return nbytes, time.perf_counter() - t0


def timed_oracle(oracle, hosts, budget_s, calib_frac=0.002):
    """The oracle on a row fraction of the sweep sized to fill about budget_s
    (calibrated on calib_frac of the rows).  Returns (GB/s, fraction, s)."""
    _, dt = oracle_sample_step(oracle, hosts, calib_frac)
    frac = min(1.0, max(1e-4, calib_frac * budget_s / max(dt, 1e-4)))
    b, t = oracle_sample_step(oracle, hosts, frac)
    return b / t / 1e9, frac, t


def cpu_baseline(hosts, budget_s=10.0, budget_1core_s=5.0):
    """The oracle timed on the host cores (OpenMP over output rows, all
    cores, then one core) on bounded samples of the sweep step."""
    import oracle
    oracle.build()
    ncpu = os.cpu_count() or 1
    oracle.set_num_threads(ncpu)
    cores = oracle.num_threads()
    v_all, f_all, t_all = timed_oracle(oracle, hosts, budget_s)
    oracle.set_num_threads(1)
    v_one, f_one, t_one = timed_oracle(oracle, hosts, budget_1core_s)
    oracle.set_num_threads(ncpu)
    return {"value": v_all, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "the first %.2f%% of the output rows of every GEMM and of every head's scored rows "
                      "in the six legs of the sweep, one pass, %.1f s" % (100 * f_all, t_all),
            "one_core": {"value": v_one, "unit": "GB/s", "cores": 1,
                         "sample": "the first %.3f%% of the rows, one pass, %.1f s" % (100 * f_one, t_one)},
            "cpu_model": cpu_model(), "nproc": ncpu}


# ----------------------------------------------------------------------------
# arms


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, timed on the host cores
    (rank 0 only), on bounded samples of the same workload."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    ncpu = os.cpu_count() or 1
    oracle.set_num_threads(ncpu)
    hosts = [host_leg(leg) for leg in LEGS]
    budget_total = 150.0
    per_step = budget_total / max(1, args.steps + args.warmup)
    _, dt = oracle_sample_step(oracle, hosts, 0.001)
    frac = min(1.0, max(1e-4, 0.001 * per_step / max(dt, 1e-4)))
    for _ in range(args.warmup):
        oracle_sample_step(oracle, hosts, frac)
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        b, t = oracle_sample_step(oracle, hosts, frac)
        tot_b += b
        tot_t += t
    value = tot_b / tot_t / 1e9
    sample = ("the first %.3f%% of the output rows of every GEMM and of every head's scored rows in the "
              "six legs of the sweep, per step" % (100 * frac))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model(), "nproc": ncpu},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def read_ceilings(torch, sv, device, stream, sizes, reps=40):
    """GB/s of the read-ceiling kernel (sv_hbm_read: only reads, same launch
    structure as the GEMMs) for each byte count, timed like the calls: back
    to back in one graph, rotating over enough buffers to exceed L2 twice."""
    out = {}
    sink = torch.empty(4096, dtype=torch.int32, device=device)
    for nb in sizes:
        copies = max(2, int(np.ceil(2 * 129 * 2 ** 20 / nb)))
        bufs = [torch.empty((nb + 15) // 16 * 16, dtype=torch.uint8, device=device) for _ in range(copies)]
        for b in bufs:
            b.fill_(1)
        fn = lambda i: sv.hbm_read(bufs[i % copies], sink, nbytes=nb // 16 * 16)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(reps):
                    fn(i)
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out[nb] = (nb // 16 * 16) * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
        del bufs, g
        torch.cuda.empty_cache()
    return out


def graph_ms(torch, g, stream, reps, rounds=3):
    """Time (ms) of one replay of graph g: the least over `rounds` runs of
    `reps` back-to-back replays, CUDA events on `stream`."""
    best = None
    for _ in range(rounds):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / reps
        best = t if best is None else min(best, t)
    return best


def time_calls_in_step(torch, sv, wl, stream, reps):
    """Each call's and each leg's time inside the step, by ablation: the
    step's graph time minus the time of the same graph without that call
    (or leg).  Events between the calls would cost each boundary the
    programmatic overlap of one kernel's tail with the next one's start
    (several microseconds), so the step is never cut; the full step is timed
    again after every ablated graph and the median taken."""
    calls = wl.calls()
    (g_full,) = wl.capture(torch, sv, [calls])
    g_full.replay()
    fulls = [graph_ms(torch, g_full, stream, reps)]
    call_ms = []
    for i in range(len(calls)):
        (g,) = wl.capture(torch, sv, [calls[:i] + calls[i + 1:]])
        g.replay()
        t = graph_ms(torch, g, stream, reps)
        fulls.append(graph_ms(torch, g_full, stream, reps))
        call_ms.append(t)
        del g
    leg_ms = []
    for l in wl.legs:
        ids = {id(c) for c in l["calls"]}
        (g,) = wl.capture(torch, sv, [[c for c in calls if id(c) not in ids]])
        g.replay()
        leg_ms.append(graph_ms(torch, g, stream, reps))
        fulls.append(graph_ms(torch, g_full, stream, reps))
        del g
    full = float(np.median(fulls))
    return ([full - t for t in call_ms], [full - t for t in leg_ms], full,
            "ablation: the step's graph time minus that of the step without the call (or leg); "
            "%d replays per timing, the least of 3 timings, the full step's median over %d timings"
            % (reps, len(fulls)))


def run_ours(args, rank, world, local_rank):
    import torch
    import speculative_verify_gb300 as sv

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    sv.load()
    wl = Workload(torch, device)
    stream = torch.cuda.current_stream(device)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    # warm-up (and the first call's scratch allocation)
    for _ in range(args.warmup):
        wl.step(sv, stream)
    torch.cuda.synchronize()
    assert sv.last_device_error() == 0

    sampler = ClockSampler(torch, device)
    sampler.start()
    # keep the GPU busy ~0.3 s before timing so clocks settle (untimed)
    t_pre = time.perf_counter()
    while time.perf_counter() - t_pre < 0.3:
        wl.step(sv, stream)
        torch.cuda.synchronize()

    calls = wl.calls()
    (g_step,) = wl.capture(torch, sv, [calls])
    for _ in range(3):
        g_step.replay()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_host0 = time.perf_counter()
    ev0.record(stream)
    for i in range(args.steps):
        g_step.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    barrier()
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms = reduce_max(dist, ms, device)
    assert sv.last_device_error() == 0

    # Inside the step: each call's and each leg's time, by ablation.
    reps = max(3, min(args.steps, 50))
    call_ms, leg_ms, full_ms, timing_how = time_calls_in_step(torch, sv, wl, stream, reps)
    call_ms = [reduce_max(dist, v, device) for v in call_ms]
    leg_ms = [reduce_max(dist, v, device) for v in leg_ms]
    assert sv.last_device_error() == 0

    # End to end through the public API with host buffers: per step the
    # activations and drafts of every call go host->device from pinned
    # memory (one copy of the input arena), the step's library calls run and
    # the verify results come back (one copy), and the host waits for them,
    # as a decode loop must before its next step.  Two ways: the copies and
    # calls captured in one CUDA graph replayed per step (a graph-capturing
    # engine), and every call made through the C ABI per step (no graph).
    in_host = wl.arena.cpu().pin_memory()
    out_host = torch.empty(wl.out.numel(), dtype=torch.int32).pin_memory()
    h2d = in_host.numel() * in_host.element_size()
    d2h = out_host.numel() * out_host.element_size()
    e2e_steps = max(1, min(args.steps, 200))
    (g_e2e,) = wl.capture(torch, sv, [calls], prologue=lambda: wl.arena.copy_(in_host, non_blocking=True),
                          epilogue=lambda: out_host.copy_(wl.out, non_blocking=True))
    out_host.fill_(-7)
    g_e2e.replay()
    torch.cuda.synchronize()
    assert int(out_host.min()) >= 0, "the end-to-end graph did not return the verify results"
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        g_e2e.replay()
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(dist, e0.elapsed_time(e1) / e2e_steps, device)
    # uncaptured: every step calls the C ABI through the binding
    out_host.fill_(-7)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        wl.arena.copy_(in_host, non_blocking=True)
        wl.step(sv, stream)
        out_host.copy_(wl.out, non_blocking=True)
        stream.synchronize()
    eager_ms = reduce_max(dist, (time.perf_counter() - t0) * 1e3 / e2e_steps, device)
    assert int(out_host.min()) >= 0
    assert sv.last_device_error() == 0

    ceilings = read_ceilings(torch, sv, device, stream, sorted({c["wbytes"] for c in calls}))
    breakdown = per_kernel_breakdown(torch, sv, device, stream) if args.breakdown else None

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    ms_per_step = ms / args.steps
    value = job_gbs(world, wl.bytes_per_step, args.steps, ms)
    # the dominant kernel: the call with the largest share of the step
    i_dom = int(np.argmax(call_ms))
    dom = calls[i_dom]
    achieved = dom["bytes"] / (call_ms[i_dom] * 1e-3) / 1e9
    clocks = sampler.summary(t_host0, t_host1)
    cpu = cpu_baseline(wl.host) if (world == 1 and not args.no_cpu_baseline) else None
    legs_out = []
    ci = 0
    for l, lm in zip(wl.legs, leg_ms):
        gbs = l["bytes"] / (lm * 1e-3) / 1e9
        cl = []
        for c in l["calls"]:
            cm = call_ms[ci]
            ci += 1
            cg = c["bytes"] / (cm * 1e-3) / 1e9
            ceil = ceilings[c["wbytes"]]
            cl.append({"call": c["label"], "kernel": kernel_of(c), "us": round(cm * 1e3, 2), "GB/s": round(cg, 1),
                       "frac_of_8TBps": round(cg / NOMINAL_HBM_GBS, 4), "frac_of_measured_copy": round(cg / peak, 4),
                       "read_ceiling": {"GB/s": round(ceil, 1), "frac": round(cg / ceil, 4)}})
        legs_out.append({"leg": l["name"], "config": l["config"], "T": l["T"], "bytes": l["bytes"],
                         "ms": round(lm, 5), "GB/s": round(gbs, 1), "frac_of_8TBps": round(gbs / NOMINAL_HBM_GBS, 4),
                         "frac_of_measured_copy": round(gbs / peak, 4), "calls": cl})
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x int4 -> fp32",
        "data": "synthetic (seeded; shapes of a 27B-class decoder)",
        "config": dict(workload_config(), parallelism="replicas" if world > 1 else "1 GPU"),
        "frac_of_8TBps": value / world / NOMINAL_HBM_GBS,
        "frac_of_measured_copy": value / world / peak,
        "legs": legs_out,
        "roofline": {"kernel": "%s (%s)" % (dom["label"], kernel_of(dom)), "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                     if peak_kind == "measured" else "fallback",
                     "algorithmic_bytes_per_launch": dom["bytes"],
                     "avg_launch_ms": call_ms[i_dom],
                     "share_of_step": call_ms[i_dom] / full_ms,
                     "traffic": recorded_traffic(dom["label"], kernel_of(dom))},
        "clocks": clocks,
        "e2e": {"value": job_gbs(world, wl.bytes_per_step, 1, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "per_step": "one CUDA graph per step holding a pinned host->device copy of every call's "
                            "activations and drafts, the step's library calls and a device->host copy of the "
                            "verify results; stream synchronize",
                "uncaptured": {"value": job_gbs(world, wl.bytes_per_step, 1, eager_ms), "unit": "GB/s",
                               "ms_per_step": eager_ms, "steps": e2e_steps,
                               "per_step": "the same copies and every library call made through the C ABI "
                                           "(ctypes binding) each step, no graph; host wall clock"}},
        "gpu_launches": wl.launches_per_step * args.steps,
        "timing": "each timed step replays one CUDA graph of the whole sweep (programmatic dependent launch "
                  "between its kernels); call and leg times inside the step: %s" % timing_how,
        "cpu_baseline": cpu,
    }
    if breakdown is not None:
        line["breakdown"] = breakdown
    print(json.dumps(line), flush=True)


def per_kernel_breakdown(torch, sv, device, stream, reps=50):
    """GB/s of each kernel alone at each T, averaged over back-to-back launches
    that rotate through enough weight copies to exceed L2 twice."""
    out = []
    rng = np.random.default_rng(99)
    l2 = 129 * 2 ** 20
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)
    cases = []
    for label, K, N in gen.GEMM_SHAPES:
        for T in (1, 4, 8, 32):
            cases.append(("gemm", label, K, N, T))
    for T, S in ((1, 1), (4, 1), (8, 1), (32, 4)):
        cases.append(("head", "lm_head", gen.HIDDEN, gen.VOCAB, (T, S)))
    for T in (1, 4):
        cases.append(("head_map", "restricted", gen.HIDDEN, gen.VOCAB, (T, 1)))
    # the greedy draft step over a full dynamic draft list (32,768 static ids
    # + 4,096 sequence tokens), and the list maintenance call itself
    cases.append(("draft_step", "list_32768+4096", gen.HIDDEN, gen.VOCAB, 1))
    # the verify whose ids are the bf16 head's: top-k of the int4 head rescored
    for k in (16, 64):
        cases.append(("head_rescored", "top%d" % k, gen.HIDDEN, gen.VOCAB, (4, k)))
    # the exact speculative sampling verify (temperature 0.7, top-k 20, top-p 0.95)
    cases.append(("head_sampled", "t0.7_k20_p0.95", gen.HIDDEN, gen.VOCAB, 4))
    cases.append(("draft_list_add", "32_tokens", 0, gen.VOCAB, 32))
    cases.append(("draft_list_add", "4096_tokens", 0, gen.VOCAB, 4096))
    for kind, label, K, N, T in cases:
        if kind == "head_rescored":
            Tt, k = T
            Wq, sc = gen.weights(rng, N, K)
            Ws = [(dev(Wq, np.int32), dev(sc, np.int16)) for _ in range(2)]
            copies = 2
            Wbf = (torch.randn((N, K), dtype=torch.float32, device=device) * 0.02).to(torch.bfloat16)
            x = dev(gen.activations(rng, Tt, K), np.int16)
            drafts = torch.zeros(Tt - 1, dtype=torch.int32, device=device)
            fn = lambda i: sv.lmhead_verify_rescored(x, Ws[i % copies][0], Ws[i % copies][1], Wbf, drafts,
                                                     top_k=k)
            # int4 head read once, plus the bf16 rows of the candidates
            nbytes = gen.lmhead_bytes(N, K, Tt, n_streams=1, n_draft=Tt - 1) + Tt * k * K * 2
            T = Tt
        elif kind == "head_sampled":
            Wq, sc = gen.weights(rng, N, K)
            Ws = [(dev(Wq, np.int32), dev(sc, np.int16)) for _ in range(2)]
            copies = 2
            x = dev(gen.activations(rng, T, K), np.int16)
            drafts = torch.zeros(T - 1, dtype=torch.int32, device=device)
            u = torch.rand(2 * T, dtype=torch.float32, device=device)
            fn = lambda i: sv.lmhead_verify_sampled(x, Ws[i % copies][0], Ws[i % copies][1], drafts, u,
                                                    temperature=0.7, top_k=20, top_p=0.95)
            nbytes = gen.lmhead_bytes(N, K, T, n_streams=1, n_draft=T - 1)
        elif kind in ("draft_step", "draft_list_add"):
            ids = rng.permutation(N).astype(np.int32)
            static = dev(ids[:32768], np.int32)
            dl = sv.DraftList(static, N, 4096)
            if kind == "draft_step":
                dl.add(dev(ids[32768:32768 + 4096], np.int32))
                Wq, sc = gen.weights(rng, N, K)
                Ws = [(dev(Wq, np.int32), dev(sc, np.int16)) for _ in range(2)]
                copies = 2
                x = dev(gen.activations(rng, 1, K), np.int16)
                a_ids = torch.empty(1, dtype=torch.int32, device=device)
                a_vals = torch.empty(1, dtype=torch.float32, device=device)
                fn = lambda i: sv.lmhead_argmax(x, Ws[i % copies][0], Ws[i % copies][1], vocab_map=dl.ids,
                                                ids=a_ids, vals=a_vals)
                nbytes = gen.lmhead_bytes(N, K, 1, n_map=32768 + 4096, n_streams=1, n_draft=0)
            else:
                # tokens that are all in the static list: every round of the
                # scan runs (worst case of one call)
                Ws = []
                toks = dev(ids[:T], np.int32)
                fn = lambda i: dl.add(toks)
                nbytes = None
        elif kind == "gemm":
            wbytes = N * K // 2
            copies = max(2, int(np.ceil(2 * l2 / wbytes)))
            Wq, sc = gen.weights(rng, N, K)
            Ws = [(dev(Wq, np.int32), dev(sc, np.int16)) for _ in range(copies)]
            x = dev(gen.activations(rng, T, K), np.int16)
            y = torch.empty((T, N), dtype=torch.bfloat16, device=device)
            fn = lambda i: sv.w4a16_gemm(x, Ws[i % copies][0], Ws[i % copies][1], y=y)
            nbytes = gen.gemm_bytes(T, K, N)
        else:
            Tt, S = T
            n_draft = Tt // S - 1
            Wq, sc = gen.weights(rng, N, K)
            Ws = [(dev(Wq, np.int32), dev(sc, np.int16)) for _ in range(2)]
            copies = 2
            x = dev(gen.activations(rng, Tt, K), np.int16)
            drafts = torch.zeros((S, n_draft), dtype=torch.int32, device=device)
            vm = dev(gen.vocab_map(rng, N, gen.DRAFT_VOCAB), np.int32) if kind == "head_map" else None
            fn = lambda i: sv.lmhead_verify_batched(x, Ws[i % copies][0], Ws[i % copies][1], drafts,
                                                    vocab_map=vm)
            n_map = gen.DRAFT_VOCAB if vm is not None else 0
            nbytes = gen.lmhead_bytes(N, K, Tt, n_map=n_map, n_streams=S, n_draft=n_draft)
            T = Tt
        for i in range(5):
            fn(i)
        torch.cuda.synchronize()
        # one graph of `reps` back-to-back launches (rotating weight copies)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for i in range(reps):
                    fn(i)
        stream.wait_stream(side)
        graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        if nbytes is None:
            out.append({"kernel": kind, "shape": label, "V": N, "tokens": T, "us": round(us, 2)})
        else:
            gbs = nbytes / (us * 1e-6) / 1e9
            out.append({"kernel": kind, "shape": label, "K": K, "N": N, "T": T, "us": round(us, 2),
                        "GB/s": round(gbs, 1), "frac_8TBps": round(gbs / NOMINAL_HBM_GBS, 3)})
        del Ws, graph
        torch.cuda.empty_cache()
    return out


def run_ncu_case(args):
    """A small, fixed workload for ncu captures: three launches of one call.
    gemm: one GEMM shape (--ncu-shape) at --ncu-T rows; head: the lm_head
    verify of --ncu-streams streams of --ncu-T / streams rows; restricted:
    the 40,960-id head at --ncu-T rows; sampled / rescored at T = 4."""
    import torch
    import speculative_verify_gb300 as sv
    sv.load()
    device = torch.device("cuda", 0)
    rng = np.random.default_rng(5)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)
    T = args.ncu_T
    if args.ncu_fma:
        sv.debug_set_fma_consumers(True)
    if args.ncu_mma_sync:
        sv.debug_set_tcgen05(False)
    if args.ncu_case == "step":
        # one warm-up step, then the profiled step: 21 launches each
        wl = Workload(torch, device)
        stream = torch.cuda.current_stream(device)
        for _ in range(2):
            wl.step(sv, stream)
        torch.cuda.synchronize()
        assert sv.last_device_error() == 0
        print(json.dumps({"ncu_case": "step", "launches_per_step": wl.launches_per_step, "ok": True}))
        return
    if args.ncu_case == "restricted":
        V, K = gen.VOCAB, gen.HIDDEN
        Wq, sc = gen.weights(rng, V, K)
        Wd, sd = dev(Wq, np.int32), dev(sc, np.int16)
        x = dev(gen.activations(rng, T, K), np.int16)
        vm = dev(gen.vocab_map(rng, V, gen.DRAFT_VOCAB), np.int32)
        drafts = torch.zeros(T - 1, dtype=torch.int32, device=device)
        for _ in range(3):
            sv.lmhead_verify_ex(x, Wd, sd, drafts.view(1, T - 1), vocab_map=vm, flags=sv.MAP_STATIC)
    elif args.ncu_case in ("head", "sampled", "rescored"):
        V, K = gen.VOCAB, gen.HIDDEN
        Wq, sc = gen.weights(rng, V, K)
        Wd, sd = dev(Wq, np.int32), dev(sc, np.int16)
        if args.ncu_case == "head":
            S = args.ncu_streams
            x = dev(gen.activations(rng, T, K), np.int16)
            drafts = torch.zeros((S, T // S - 1), dtype=torch.int32, device=device)
            for _ in range(3):
                sv.lmhead_verify_batched(x, Wd, sd, drafts)
        else:
            T = 4
            x = dev(gen.activations(rng, T, K), np.int16)
            drafts = torch.zeros(T - 1, dtype=torch.int32, device=device)
            if args.ncu_case == "sampled":
                u = torch.rand(2 * T, dtype=torch.float32, device=device)
                for _ in range(3):
                    sv.lmhead_verify_sampled(x, Wd, sd, drafts, u, temperature=0.7, top_k=20, top_p=0.95)
            else:
                Wbf = (torch.randn((V, K), dtype=torch.float32, device=device) * 0.02).to(torch.bfloat16)
                for _ in range(3):
                    sv.lmhead_verify_rescored(x, Wd, sd, Wbf, drafts, top_k=16)
    else:
        label, K, N = {s[0]: s for s in gen.GEMM_SHAPES}[args.ncu_shape]
        Wq, sc = gen.weights(rng, N, K)
        Wd, sd = dev(Wq, np.int32), dev(sc, np.int16)
        x = dev(gen.activations(rng, T, K), np.int16)
        for _ in range(3):
            sv.w4a16_gemm(x, Wd, sd)
    torch.cuda.synchronize()
    assert sv.last_device_error() == 0
    print(json.dumps({"ncu_case": args.ncu_case, "T": T, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--breakdown", action="store_true", help="also time each kernel alone at T=1..32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", choices=["head", "gemm", "sampled", "rescored", "restricted", "step"], default=None)
    ap.add_argument("--ncu-fma", action="store_true", help="CUDA-core consumers (sv_debug_set_fma_consumers)")
    ap.add_argument("--ncu-mma-sync", action="store_true",
                    help="the mma.sync stream kernel for 17..32 tokens (sv_debug_set_tcgen05(0))")
    ap.add_argument("--ncu-T", type=int, default=4)
    ap.add_argument("--ncu-streams", type=int, default=1)
    ap.add_argument("--ncu-shape", choices=[s[0] for s in gen.GEMM_SHAPES], default="gate_up")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.ncu_case:
        run_ncu_case(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
