#!/usr/bin/env python3
"""Benchmark of the batched RNS-NTT hot path on GB300.

One step = every kernel of the hot path once, chained on the n = 2^16, L = 24
workload (16 polynomials = 4 pairs of 2-component ciphertexts, 201 MB of u64
residues; key switch over 24 + 8 primes with dnum = 3):

  1. fhe_ntt_fwd      X[2][4][2][24][n]           coefficient -> NTT   (384 transforms)
                      (X[0]: the 4 ciphertexts a, X[1]: the 4 ciphertexts b)
  2. fhe_automorph    Y = sigma_k(X)  NTT domain  k = 5^(2^(step mod 16)) mod 2n
  3. fhe_mul_ntt      Z = X * Y
  4. fhe_tensor       D[4][3][24][n] = tensor(Z[0], Z[1])
  5. fhe_ntt_inv      D                           NTT -> coefficient   (288 transforms)
  6. fhe_keyswitch_ip KS[4][2][32][n] = keyswitch(D[:, 2])  (ModUp + 384 transforms + IP)

metric: NTT (poly x prime)/s = 1056 transforms per step / step time (whole
job, inputs resident in HBM).  Per-kernel CUDA-event times give the NTT's
achieved GB/s and the key-switch ops/s.  `--impl reference` times the CPU
oracle on a bounded sample of the same step instead.
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LOG_N, N, L, K, DNUM, PAIRS = 16, 1 << 16, 24, 8, 3, 4
NPOLY = PAIRS * 2 * 2                      # 16 polynomials
FWD_T, INV_T, KS_T = NPOLY * L, PAIRS * 3 * L, PAIRS * DNUM * (L + K)
UNITS = FWD_T + INV_T + KS_T               # 1056 poly x prime NTTs per step
METRIC = "NTT (poly×prime)/s and achieved GB/s at n=2^16,L=24; key-switch ops/s"
UNIT = "NTT (poly x prime)/s"
WORKLOAD = "n=2^16, L=24 primes (largest q<2^50, q=1 mod 2^17), 16 polys = 4 ciphertext pairs; " \
           "fwd NTT -> automorph -> mul -> tensor -> inv NTT -> key switch (24+8 primes, dnum=3) x4"
# Integer-pipe roofline of one lazy Shoup butterfly (3 mul.wide + 2 mul.hi +
# 4 mul.lo on the FMA pipe; measured pipe rates on GB300: 25.2, 32 and 64 per
# clock per SM), at the maximum SM clock.
BFLY_PER_CLK_SM = 1.0 / (3 / 25.2 + 2 / 32.0 + 4 / 64.0)
SMS, SM_MAX_MHZ = 152, 2070.0
ALU_PEAK_BFLY = SMS * BFLY_PER_CLK_SM * SM_MAX_MHZ * 1e6
BFLY_PER_FWD = NPOLY * L * (N // 2) * LOG_N
BFLY_PER_INV = INV_T * (N // 2) * LOG_N
NTT_BYTES_PER_FWD = 16 * NPOLY * L * N     # read + write every residue once
NTT_BYTES_PER_INV = 16 * INV_T * N
KS_MIN_BYTES_X4 = 8 * N * (PAIRS * (L + 2 * (L + K)) + DNUM * 2 * (L + K))   # 285.2 MB


def keyswitch_alu_floor_s(pairs: int = PAIRS) -> float:
    """Seconds the integer multiply pipe needs for `pairs` key switches of the
    bench shape if it did nothing else: every 32-bit product the kernels
    execute on it, at the pipe's measured per-SM rates (low 64, high 32, wide
    25.2 per clock) on 152 SMs at the maximum clock -- the same derivation as
    ALU_PEAK_BFLY.  Lazy Shoup product (butterfly, CRT bracket): 3 wide +
    2 high + 4 low; fixed-point term of the correction count (64 x 16-bit low
    product + 64 x 64 high product): 4 wide + 1 high + 1 low; 64-bit Barrett
    step with a 16-bit mu: 2 wide + 1 high + 1 low; multiply-accumulate of
    25-bit halves: 3 wide; reduction of a 105-bit sum: 5 wide + 2 high + 3 low.
    Per (coefficient, digit) the tensor-core ModUp does alpha brackets, alpha
    fixed-point terms and one Barrett step per target (its dot products run on
    the tensor cores, KS_TENSOR_FLOP); per output residue of the inner product:
    2 dnum multiply-accumulates and 2 reductions."""
    lo, hi, wide = 1 / 64.0, 1 / 32.0, 1 / 25.2          # SM-cycles per 32-bit product
    shoup, mac, red = 3 * wide + 2 * hi + 4 * lo, 3 * wide, 5 * wide + 2 * hi + 3 * lo
    fixp, barrett = 4 * wide + hi + lo, 2 * wide + hi + lo
    alpha = L // DNUM
    targets = L + K - alpha
    bfly = pairs * DNUM * (L + K) * (N // 2) * LOG_N
    units = pairs * DNUM * N
    ip = pairs * (L + K) * N
    cycles = (bfly * shoup + units * (alpha * (shoup + fixp) + targets * barrett)
              + ip * (2 * DNUM * mac + 2 * red))
    return cycles / (SMS * SM_MAX_MHZ * 1e6)


# fp16 tensor-core work of the tensor-core ModUp per call: every tile of 128
# coefficients of a digit is a 128 x (8 targets) x (8 alpha) product (targets in
# groups of 16, N padded to a multiple of 16), 2 flops per multiply-add.
KS_TENSOR_FLOP = 2 * PAIRS * DNUM * N * (8 * (L + K - L // DNUM)) * (8 * (L // DNUM))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_traffic(key: str, rows_per_launch: int):
    """DRAM bytes (read + write) per launch of a kernel from the committed ncu
    capture, or None when the kernel's source has changed since it was taken
    or the capture was of another launch size."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[key]
        h = hashlib.sha256()
        for path in rec["source_files"]:
            with open(os.path.join(ROOT, path), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != rec["source_sha256_16"] or rec["rows_per_launch"] != rows_per_launch:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


TRAFFIC_SOURCE = ("dram__bytes_read.sum + dram__bytes_write.sum of the launches of one call, from the committed ncu "
                  "capture that profiles/traffic.json names; null when the kernels' sources changed since that capture")


def ntt_fwd_traffic():
    return kernel_traffic("k_ntt_fwd", NPOLY * L)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(rank: int) -> int:
    """Each rank transforms its own shard of ciphertexts (weak scaling, no
    data exchange): rank r draws its inputs from seed 3 + 1000 r."""
    return 3 + 1000 * rank


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank time over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, max_ms: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    return units_per_rank * world / (max_ms * 1e-3)


# --------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        load = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ our arm ------

class NvmlClockPoller:
    """SM clock, clock-event reasons and power read through NVML (read-only
    queries, no setting is changed) every `period` seconds by a thread, for
    exactly the span between start() and stop(): the timed region itself,
    which is too short for nvidia-smi's 100 ms sampling.  `reader` replaces
    NVML (tests); it returns (sm_mhz, max_sm_mhz, reason_bits, power_mw)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device=None, period: float = 0.002, reader=None):
        import threading
        self.period, self.samples, self._stop = period, [], threading.Event()
        self._thread = None
        self.reader = reader or self._nvml_reader(device)

    @staticmethod
    def _nvml_reader(device):
        import ctypes
        try:
            import torch
            props = torch.cuda.get_device_properties(device)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                return None
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:   # NVML_CLOCK_SM
                return None
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            return None

        def read():
            clk, rs, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
            nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
            reasons_fn(h, ctypes.byref(rs))
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
            return clk.value, mx.value, rs.value, mw.value
        return read

    def start(self):
        import threading
        if self.reader is None:
            return self

        def loop():
            while not self._stop.is_set():
                self.samples.append(self.reader())
                time.sleep(self.period)
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        return self

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self.samples.append(self.reader())   # at least one sample at the end of the region

    def summary(self):
        if not self.samples:
            return None
        sm = [c for c, _, _, _ in self.samples]
        bits = 0
        for _, _, r, _ in self.samples:
            bits |= r
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(m for _, m, _, _ in self.samples),
                "sm_min_mhz": min(sm), "reasons": sorted(n for b, n in self.REASONS.items() if bits & b),
                "samples": len(self.samples), "power_w_max": max(p for _, _, _, p in self.samples) / 1000.0,
                "source": f"NVML every {self.period * 1e3:g} ms inside the timed region"}


def clock_record(poller, sampler):
    """The NVML record of the timed region when NVML was readable, else nvidia-smi's."""
    rec = poller.summary() if poller is not None else None
    return rec if rec is not None else sampler.summary()


def build_state(device, seed: int = 3):
    import torch
    from ntt_arithmetic_gb300 import api, inputs
    q = api.find_primes(LOG_N, L)
    p = api.find_primes(LOG_N, K, below=q[-1])
    qp = q + p
    st = {"q": q, "qp": qp}
    st["tq"] = api.NttTables(LOG_N, q, device)
    st["tqp"] = api.NttTables(LOG_N, qp, device)
    st["modup"] = api.ModupTables(L, K, DNUM, qp, device)
    x_host = inputs.uniform_residues((2, PAIRS, 2, L, N), q, seed=seed, buffer=0)
    keys_host = inputs.uniform_residues((DNUM, 2, L + K, N), qp, seed=seed, buffer=1)
    st["x_pinned"] = torch.from_numpy(x_host).pin_memory()
    st["X"] = st["x_pinned"].to(device)
    st["keys"] = torch.from_numpy(keys_host).to(device)
    st["Y"] = torch.empty_like(st["X"])
    st["D"] = torch.empty((PAIRS, 3, L, N), dtype=torch.uint64, device=device)
    st["KS"] = torch.empty((PAIRS, 2, L + K, N), dtype=torch.uint64, device=device)
    st["ws"] = torch.empty(api.keyswitch_workspace_bytes(LOG_N, L, K, DNUM, PAIRS) // 8, dtype=torch.uint64,
                           device=device)
    st["ks_pinned"] = torch.empty(st["KS"].shape, dtype=torch.uint64).pin_memory()
    return st


def butterfly_ceiling(st, device, reps: int = 5) -> float:
    """Butterflies/s of the library's register-resident butterfly probe
    (fhe_butterfly_probe: the NTT's butterfly with no memory traffic), 4 waves
    of 2 CTAs per SM, median of `reps` launches timed with CUDA events."""
    import torch
    from ntt_arithmetic_gb300 import api
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    out = torch.empty(sms * 2 * 4 * 256, dtype=torch.uint64, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(2):
        api.butterfly_probe(out, 64, st["tq"])
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bfly = api.butterfly_probe(out, 64, st["tq"])
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    return bfly / statistics.median(times)


def run_step(st, step: int, ev=None, X=None, KS=None):
    """One pass of the hot path on input X (default st["X"]) into KS
    (default st["KS"]); `ev` (list of 7 events) brackets each call."""
    from ntt_arithmetic_gb300 import api
    k = pow(5, 1 << (step % 16), 2 * N)
    rec = (lambda i: ev[i].record()) if ev else (lambda i: None)
    X = st["X"] if X is None else X
    KS = st["KS"] if KS is None else KS
    Y, D = st["Y"], st["D"]
    rec(0)
    api.ntt_fwd(X, st["tq"])
    rec(1)
    api.automorph(Y, X, k, st["tq"], domain="ntt")
    rec(2)
    api.mul_ntt(Y, X, Y, st["tq"])
    rec(3)
    api.tensor(D, Y[0], Y[1], st["tq"])
    rec(4)
    api.ntt_inv(D, st["tq"])
    rec(5)
    # relinearisation input: component d2 of each of the 4 products (batch stride 3 L n)
    api.keyswitch_ip(KS, D, st["keys"], L, K, DNUM, st["tqp"], st["modup"], st["ws"],
                     in_offset=2 * L * N, in_stride=3 * L * N, batch=PAIRS)
    rec(6)


def run_step_halves(st, step: int, streams):
    """The same step as run_step, as two independent halves of 2 ciphertext
    pairs each, one per stream: the halves' kernels may run at the same time,
    so one half's HBM-bound kernels (automorphism, products) can share the
    SMs with the other half's integer-pipe-bound ones (NTT, ModUp)."""
    from ntt_arithmetic_gb300 import api
    k = pow(5, 1 << (step % 16), 2 * N)
    X, Y, D, KS = st["X"], st["Y"], st["D"], st["KS"]
    h = PAIRS // 2
    wsh = st["ws"].view(PAIRS, -1)
    for i, s in enumerate(streams):
        sl = slice(i * h, (i + 1) * h)
        for a in range(2):
            api.ntt_fwd(X[a, sl], st["tq"], stream=s)
        for a in range(2):
            api.automorph(Y[a, sl], X[a, sl], k, st["tq"], domain="ntt", stream=s)
            api.mul_ntt(Y[a, sl], X[a, sl], Y[a, sl], st["tq"], stream=s)
        api.tensor(D[sl], Y[0, sl], Y[1, sl], st["tq"], stream=s)
        api.ntt_inv(D[sl], st["tq"], stream=s)
        api.keyswitch_ip(KS[sl], D[sl], st["keys"], L, K, DNUM, st["tqp"], st["modup"], wsh[sl].reshape(-1),
                         stream=s, in_offset=2 * L * N, in_stride=3 * L * N, batch=h)


def two_stream_ms(st, steps: int, warmup: int, device) -> float:
    """Mean ms per step of run_step_halves, between events on the main
    stream that both halves' streams wait for / are waited on."""
    import torch
    main = torch.cuda.current_stream(device)
    streams = [torch.cuda.Stream(device), torch.cuda.Stream(device)]

    def one(i):
        ev = torch.cuda.Event()
        ev.record(main)
        for s in streams:
            s.wait_event(ev)
        run_step_halves(st, i, streams)
        for s in streams:
            done = torch.cuda.Event()
            done.record(s)
            main.wait_event(done)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    for i in range(steps):
        one(warmup + i)
    b.record(main)
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) / steps


def e2e_steps(st, steps: int, device) -> float:
    """Mean ms per step end to end: every step copies its input X from pinned
    host memory and reads its key-switch output back to pinned host memory.
    The copies run on their own streams, double-buffered, so step i's input
    copy and step i-1's output copy overlap step i-1's and step i's kernels
    (a serving pipeline); events order every buffer reuse."""
    import torch
    # three non-default streams: the legacy default stream would serialise
    # with the copy streams
    comp, s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    if "X2" not in st:
        st["X2"] = torch.empty_like(st["X"])
        st["KS2"] = torch.empty_like(st["KS"])
        st["ks_pinned2"] = torch.empty(st["KS"].shape, dtype=torch.uint64).pin_memory()
    Xb, KSb, outb = [st["X"], st["X2"]], [st["KS"], st["KS2"]], [st["ks_pinned"], st["ks_pinned2"]]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]     # step's kernels finished with X[b] and KS[b]
    ev_out = [torch.cuda.Event() for _ in range(2)]      # KS[b] copied out
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    start.record(comp)
    for e in ev_done + ev_out:
        e.record(comp)
    for i in range(steps):
        b = i % 2
        s_in.wait_event(start)
        s_in.wait_event(ev_done[b])              # X[b] no longer read by step i-2
        with torch.cuda.stream(s_in):
            Xb[b].copy_(st["x_pinned"], non_blocking=True)
        ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        comp.wait_event(ev_out[b])               # KS[b] of step i-2 copied out
        with torch.cuda.stream(comp):
            run_step(st, i, X=Xb[b], KS=KSb[b])
        ev_done[b].record(comp)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            outb[b].copy_(KSb[b], non_blocking=True)
        ev_out[b].record(s_out)
    for e in ev_out:
        comp.wait_event(e)
    stop.record(comp)
    torch.cuda.synchronize(device)
    return start.elapsed_time(stop) / steps


def ours(args):
    import torch
    import torch.distributed as dist
    from ntt_arithmetic_gb300 import api
    from ntt_arithmetic_gb300 import build as B
    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(B.OUT):
        B.build()
    if ws > 1:
        dist.barrier()
    st = build_state(device, rank_seed(rank))
    stream = torch.cuda.current_stream(device)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    for i in range(args.warmup):
        run_step(st, i)
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = api.launch_count()
    with ClockSampler(local) as clk:
        barrier()
        poll = NvmlClockPoller(device).start()
        start.record(stream)
        for i in range(args.steps):
            run_step(st, args.warmup + i)
        stop.record(stream)
        barrier()
        launches = api.launch_count() - launches0
        # the same steps again with an event between calls, for the per-call times the rooflines use
        # (an event between two calls also ends the early placement of the second call's CTAs)
        for i in range(args.steps):
            run_step(st, args.warmup + args.steps + i, evs[i])
        barrier()
        poll.stop()
    ms = start.elapsed_time(stop) / args.steps
    per = [[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(6)] for i in range(args.steps)]
    kern = [statistics.mean(p[j] for p in per) for j in range(6)]
    ms_max = max_over_ranks(ms, device)

    # end to end through the public API with host buffers: every step copies
    # its input from pinned host memory and its key-switch output back
    barrier()
    e2e_steps(st, max(3, args.warmup), device)          # warm-up of the copy pipeline (streams, pinned buffers)
    e2e_ms = max_over_ranks(e2e_steps(st, args.steps, device), device)
    # the same work as two concurrent halves on two streams (reported beside the main figure)
    barrier()
    two_ms = max_over_ranks(two_stream_ms(st, args.steps, max(3, args.warmup), device), device)

    clocks = clock_record(poll, clk)
    hbm, hbm_kind = peaks()
    fwd_s, inv_s, ks_s = kern[0] * 1e-3, kern[4] * 1e-3, kern[5] * 1e-3
    achieved_bfly = BFLY_PER_FWD / fwd_s
    achieved_inv = BFLY_PER_INV / inv_s
    ceiling = butterfly_ceiling(st, device)   # outside the timed region
    ks_alu_s = keyswitch_alu_floor_s()
    ks_hbm_s = KS_MIN_BYTES_X4 / (hbm * 1e9)
    line = {
        "metric": METRIC,
        "value": whole_job_rate(UNITS, ws, ms_max),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u64",
        "data": "synthetic: seeded uniform residues in [0, q) (SplitMix64 counter generator)",
        "config": {"workload": WORKLOAD, "n": N, "L": L, "K": K, "dnum": DNUM, "polys": NPOLY,
                   "units_per_step": UNITS, "l2": "inputs larger than L2 (201 MB residues + 101 MB keys per step)",
                   "parallelism": f"replicas x{ws}"},
        "kernels_ms": {"ntt_fwd": kern[0], "automorph_ntt": kern[1], "mul_ntt": kern[2], "tensor": kern[3],
                       "ntt_inv": kern[4], "keyswitch_ip_x4": kern[5]},
        "ntt_fwd_gbs": NTT_BYTES_PER_FWD / fwd_s / 1e9,
        "ntt_fwd_poly_prime_per_s": NPOLY * L / fwd_s,
        "ntt_fwd_hbm_frac": NTT_BYTES_PER_FWD / fwd_s / 1e9 / hbm,
        "keyswitch_ops_per_s": PAIRS / (kern[5] * 1e-3) * ws,
        # fully fused minimum of the step's 4 key switches: 4 inputs [24][n] + the shared keys
        # [3][2][32][n] + 4 outputs [2][32][n], 8 B each, in the measured time, against the HBM peak
        "keyswitch_x4_hbm_bound_frac": (KS_MIN_BYTES_X4 / (kern[5] * 1e-3) / 1e9) / hbm,
        "roofline": {"bound": "alu", "achieved": achieved_bfly / 1e9, "peak": ALU_PEAK_BFLY / 1e9,
                     "unit": "Gbutterfly/s", "frac": achieved_bfly / ALU_PEAK_BFLY, "traffic": ntt_fwd_traffic(),
                     "traffic_unit": "bytes/launch", "traffic_source": TRAFFIC_SOURCE,
                     "algorithmic_bytes": NTT_BYTES_PER_FWD,
                     "kernel": "forward NTT call = k_ntt_fwd_cols<16,6,3> (first 6 stages, strided columns) + "
                               "k_ntt_fwd_blk<16,6,6,4,10> (last 10 stages, one CTA per 1024-residue block); "
                               "n=2^16, 384 rows; traffic = both launches",
                     "peak_kind": "derived: measured integer-pipe rates x 152 SMs x 2070 MHz",
                     "measured_butterfly_ceiling": ceiling / 1e9, "frac_of_measured_ceiling": achieved_bfly / ceiling,
                     "ceiling_note": "fhe_butterfly_probe: the same butterfly register-resident, no memory traffic",
                     "hbm_gbs": NTT_BYTES_PER_FWD / fwd_s / 1e9, "hbm_peak_gbs": hbm, "hbm_peak_kind": hbm_kind,
                     "hbm_frac": NTT_BYTES_PER_FWD / fwd_s / 1e9 / hbm,
                     "hbm_frac_bound_at_ceiling": NTT_BYTES_PER_FWD / (BFLY_PER_FWD / ceiling) / 1e9 / hbm},
        "roofline_ntt_inv": {"bound": "alu", "achieved": achieved_inv / 1e9, "peak": ALU_PEAK_BFLY / 1e9,
                             "unit": "Gbutterfly/s", "frac": achieved_inv / ALU_PEAK_BFLY,
                             "traffic": kernel_traffic("k_ntt_inv", INV_T), "traffic_unit": "bytes/launch",
                             "traffic_source": TRAFFIC_SOURCE,
                             "algorithmic_bytes": NTT_BYTES_PER_INV,
                             "kernel": "inverse NTT call = k_ntt_inv_blk<16,6,6,4,8> (first 10 stages per block) + "
                                       "k_ntt_inv_cols<16,6,3> (last 6 stages and the twist n^-1 psi^-j); n=2^16, "
                                       "288 rows; traffic = both launches",
                             "frac_of_measured_ceiling": achieved_inv / ceiling,
                             "hbm_gbs": NTT_BYTES_PER_INV / inv_s / 1e9, "hbm_frac": NTT_BYTES_PER_INV / inv_s / 1e9 / hbm,
                             "poly_prime_per_s": INV_T / inv_s},
        "roofline_keyswitch": {"bound": "alu" if ks_alu_s >= ks_hbm_s else "hbm",
                               "achieved": PAIRS / ks_s, "peak": PAIRS / max(ks_alu_s, ks_hbm_s),
                               "unit": "key switches/s", "frac": max(ks_alu_s, ks_hbm_s) / ks_s,
                               "alu_floor_ms": ks_alu_s * 1e3, "hbm_floor_ms": ks_hbm_s * 1e3, "measured_ms": ks_s * 1e3,
                               "frac_alu_at_measured_ceiling": ks_alu_s * (ALU_PEAK_BFLY / ceiling) / ks_s,
                               "hbm_bytes_min": KS_MIN_BYTES_X4,
                               "traffic": kernel_traffic("keyswitch", KS_T), "traffic_unit": "bytes/call",
                               "traffic_source": TRAFFIC_SOURCE,
                               "tensor_flop": KS_TENSOR_FLOP,
                               "work": "4 key switches of [24][n] over 24 + 8 primes, dnum = 3: ModUp (8 CRT brackets, 8 "
                                       "fixed-point terms and 24 Barrett steps per coefficient and digit on the integer "
                                       "pipes; the extension's 128 x 192 x 64 fp16 products per tile of 128 "
                                       "coefficients on the tensor cores), 384 NTT rows, inner product (6 "
                                       "multiply-accumulates + 2 reductions per output residue); HBM floor: inputs + "
                                       "keys (read once) + outputs"},
        "clocks": clocks,
        "gpu_launches": launches,
        "two_streams": {"value": whole_job_rate(UNITS, ws, two_ms), "unit": UNIT, "ms_per_step": two_ms,
                        "note": "the step's 4 ciphertext pairs as two independent halves of 2, each on its own "
                                "stream, so that one half's HBM-bound kernels overlap the other's integer-bound "
                                "ones; the line's value and kernel times are the one-stream step's"},
        "e2e": {"value": whole_job_rate(UNITS, ws, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms, "steps": args.steps,
                "h2d_bytes_per_step": st["x_pinned"].numel() * 8, "d2h_bytes_per_step": st["ks_pinned"].numel() * 8,
                "pipelining": "input/output copies on their own streams, double-buffered across steps"},
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_sample_steps)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


# ------------------------------------------------------- oracle (CPU) arm --

def oracle_sample_state():
    """One of the 4 ciphertext pairs of the step (a quarter of its work)."""
    import oracle
    from ntt_arithmetic_gb300 import inputs
    qp = [int(v) for v in oracle.primes(2 * N, L + K)]
    q = qp[:L]
    x = inputs.uniform_residues((2, PAIRS, 2, L, N), q, seed=3, buffer=0)[:, :1]
    keys = inputs.uniform_residues((DNUM, 2, L + K, N), qp, seed=3, buffer=1)
    return {"q": q, "qp": qp, "psi_q": oracle.psis(q, N), "psi_qp": oracle.psis(qp, N), "x": x, "keys": keys}


def oracle_step(s, step: int, threads: int):
    import oracle
    k = pow(5, 1 << (step % 16), 2 * N)
    X = oracle.ntt_batch(s["x"], s["q"], s["psi_q"], threads=threads)
    Y = oracle.automorph_batch(X, s["q"], s["psi_q"], k, ntt_domain=True, threads=threads)
    Z = oracle.mul_batch(X, Y, s["q"])
    D = oracle.tensor_batch(Z[0], Z[1], s["q"])
    D = oracle.ntt_batch(D, s["q"], s["psi_q"], inverse=True, threads=threads)
    oracle.keyswitch_batch(D[:, 2], s["keys"], s["qp"], s["psi_qp"], L, K, DNUM, threads=threads)


SAMPLE_UNITS = UNITS // PAIRS   # transforms in one pair's share of the step


def cpu_baseline(steps: int):
    import oracle
    threads = oracle.default_threads()
    s = oracle_sample_state()
    t0 = time.perf_counter()
    for i in range(steps):
        oracle_step(s, i, threads)
    dt = (time.perf_counter() - t0) / steps
    t0 = time.perf_counter()
    oracle_step(s, 0, 1)                      # the same sample on one core, once
    dt1 = time.perf_counter() - t0
    return {"value": SAMPLE_UNITS / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"1 of the 4 ciphertext pairs of the step ({SAMPLE_UNITS} transforms + its automorph, "
                      f"mul, tensor and 1 key switch), {steps} step(s), {dt:.2f} s/step, {threads} threads",
            "single_thread": {"value": SAMPLE_UNITS / dt1, "unit": UNIT, "cores": 1, "s_per_step": dt1}}


def reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from oracle import build as OB
    OB.build() if OB.stale() else None
    threads = oracle.default_threads()
    s = oracle_sample_state()
    for i in range(args.warmup):
        oracle_step(s, i, threads)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(s, args.warmup + i, threads)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = SAMPLE_UNITS / dt
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u64",
        "data": "synthetic: seeded uniform residues in [0, q) (SplitMix64 counter generator)",
        "config": {"workload": WORKLOAD, "n": N, "L": L, "K": K, "dnum": DNUM, "polys": NPOLY,
                   "units_per_step": SAMPLE_UNITS, "sample": "1 of 4 ciphertext pairs per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"1 of the 4 ciphertext pairs of the step per timed step, {threads} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def sweep(args):
    """Per-point times of the sweep workload (n = 2^11..2^17, L in {1, 8, 24,
    64}, batch in {1, 16, 64}): forward NTT, inverse NTT and pointwise product,
    each timed with CUDA events on the launch stream after 3 warm-up runs,
    with L2 flushed (256 MB write) before every timed repetition.  One JSON
    line per point; these are measurements, not the headline bench line."""
    import torch
    from ntt_arithmetic_gb300 import api, inputs
    from ntt_arithmetic_gb300 import build as B
    B.build()
    dev = torch.device("cuda", 0)
    hbm, hbm_kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for log_n in range(11, 18):
        n = 1 << log_n
        for L in (1, 8, 24, 64):
            qs = api.find_primes(log_n, L)
            t = api.NttTables(log_n, qs, dev)
            pool = torch.from_numpy(inputs.uniform_residues((2, L, n), qs, 5000 + log_n, buffer=L)).to(dev)
            for batch in (1, 16, 64):
                x = pool.repeat((batch + 1) // 2, 1, 1)[:batch].contiguous()
                y = x.clone()
                times = {"fwd": [], "inv": [], "mul": []}
                for rep in range(3 + args.sweep_reps):
                    for name in ("fwd", "inv", "mul"):
                        flush.zero_()
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        if name == "fwd":
                            api.ntt_fwd(x, t)
                        elif name == "inv":
                            api.ntt_inv(x, t)
                        else:
                            api.mul_ntt(x, x, y, t)
                        e1.record(stream)
                        torch.cuda.synchronize(dev)
                        if rep >= 3:
                            times[name].append(e0.elapsed_time(e1) * 1e3)
                med = {k: statistics.median(v) for k, v in times.items()}
                residues = batch * L * n
                bfly = batch * L * (n // 2) * log_n
                print(json.dumps({
                    "sweep_point": {"n": n, "L": L, "batch": batch}, "bytes": residues * 8,
                    "fwd_us": round(med["fwd"], 2), "inv_us": round(med["inv"], 2), "mul_us": round(med["mul"], 2),
                    "fwd_gbs": round(16 * residues / med["fwd"] / 1e3, 1), "inv_gbs": round(16 * residues / med["inv"] / 1e3, 1),
                    "mul_gbs": round(24 * residues / med["mul"] / 1e3, 1),
                    "fwd_hbm_frac": round(16 * residues / med["fwd"] / 1e3 / hbm, 3),
                    "mul_hbm_frac": round(24 * residues / med["mul"] / 1e3 / hbm, 3),
                    "fwd_alu_frac": round(bfly / (med["fwd"] * 1e-6) / ALU_PEAK_BFLY, 3),
                    "hbm_peak_gbs": hbm, "hbm_peak_kind": hbm_kind, "l2": "flushed before every timed run"}), flush=True)
                del x, y
            torch.cuda.empty_cache()


# ------------------------------------------------- widened rows of the path --
#
# Each workload below is one more part of the key-switch / bootstrap path,
# timed with the same rules as the headline step: warm-up, CUDA events on the
# launch stream around exactly `steps` iterations with inputs larger than L2,
# clocks sampled during the timed region, a live-timed roofline for the
# row's dominant kernel, an end-to-end number with host buffers, and the
# oracle on a bounded sample as the CPU baseline.

SHOUP_PER_CLK_SM = BFLY_PER_CLK_SM        # a lazy Shoup product costs what a butterfly's multiply does
ALU_PEAK_SHOUP = ALU_PEAK_BFLY


def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _time_calls(fn, reps: int, warm: int = 3) -> float:
    """Mean ms of `fn` over `reps` back-to-back calls on the current stream."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = _events(2)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _rand_dev(shape_lead, mods, n, seed, dev):
    import torch
    from ntt_arithmetic_gb300 import inputs
    return torch.from_numpy(inputs.uniform_residues(tuple(shape_lead) + (len(mods), n), mods, seed, buffer=7)).to(dev)


class RowBench:
    """One widened workload: subclasses fill in the state, the step, the
    dominant kernel's probe and the oracle sample."""
    name = metric = unit = workload = ""
    units_per_step = 1
    l2 = "inputs larger than L2"

    def setup(self, dev):
        raise NotImplementedError

    def step(self):
        raise NotImplementedError

    def before_step(self):
        """Untimed work between timed steps (an L2 flush for inputs smaller than L2)."""

    def probe(self):
        """(callable launching the dominant kernel once, roofline dict sans achieved/frac)."""
        raise NotImplementedError

    def e2e_step(self):
        """One step through the public API with the H2D copy of its input and
        the D2H copy of its result; returns (h2d bytes, d2h bytes)."""
        raise NotImplementedError

    def oracle_setup(self):
        """Host inputs of the oracle sample (oracle primes + the seeded generator only)."""
        raise NotImplementedError

    def oracle_sample(self):
        """(seconds, units of the metric done, description) for a bounded sample."""
        raise NotImplementedError

    def config(self):
        return {"workload": self.workload, "l2": self.l2}

    def replayed_launches(self, steps):
        """Kernels launched by CUDA-graph replays in `steps` timed steps (the
        library's launch counter sees only direct calls)."""
        return 0


class ModdownRow(RowBench):
    name = "moddown"
    metric = "ModDown (QP->Q) polys/s, NTT domain, n=2^16, 24+8 primes"
    unit = "poly/s"
    workload = ("ModDown of the 4 key-switch outputs KS[4][2][32][n] of the headline step (NTT domain, nearest "
                "rounding, P = 8 primes) -> [4][2][24][n]; n=2^16")
    units_per_step = 8
    traffic_rows = 8 * L         # output rows of the captured call

    def setup(self, dev):
        import torch
        from ntt_arithmetic_gb300 import api
        q = api.find_primes(LOG_N, L)
        self.qp = q + api.find_primes(LOG_N, K, below=q[-1])
        self.t = api.NttTables(LOG_N, self.qp, dev)
        self.md = api.ModdownTables(L, K, self.qp, dev)
        self.x = _rand_dev((8,), self.qp, N, 31, dev)
        self.out = torch.empty((8, L, N), dtype=torch.uint64, device=dev)
        self.ws = torch.empty(api.moddown_workspace_bytes(LOG_N, L, K, 8) // 8, dtype=torch.uint64, device=dev)
        self.x_pin = self.x.cpu().pin_memory()
        self.o_pin = torch.empty(self.out.shape, dtype=torch.uint64).pin_memory()

    def step(self):
        from ntt_arithmetic_gb300 import api
        api.moddown(self.out, self.x, L, K, self.t, self.md, domain="ntt", nearest=True, workspace=self.ws)

    def probe(self):
        # the row's own call, against the integer-pipe floor of its products, in units of one lazy Shoup
        # product (the butterfly peak's unit): the inverse NTT of the 8 x 8 rows of P limbs and the forward
        # NTT of the 8 x 24 rows of d (one Shoup product per butterfly), the tensor-core conversion's K CRT
        # brackets, K fixed-point terms and L Barrett steps per coefficient, and one Shoup product per output
        lo, hi, wide = 1 / 64.0, 1 / 32.0, 1 / 25.2
        shoup = 3 * wide + 2 * hi + 4 * lo
        fixp, barrett = 4 * wide + hi + lo, 2 * wide + hi + lo
        bfly = 8 * (K + L) * (N // 2) * LOG_N
        conv = 8 * N * (K * (shoup + fixp) + L * barrett) / shoup
        final = 8 * L * N
        ops = bfly + conv + final
        fn = self.step
        return fn, {"bound": "alu", "work": ops, "peak": ALU_PEAK_SHOUP / 1e9, "unit": "G Shoup-product equivalents/s",
                    "kernel": "one NTT-domain ModDown call, batch 8: k_ntt_inv_blk + k_ntt_inv_cols (64 rows of P "
                              "limbs), k_moddown_tc (conversion on the tensor cores), k_ntt_fwd_cols + "
                              "k_ntt_fwd_blk_md (192 rows of d + the last product)",
                    "work_note": (f"{bfly / 1e6:.1f} M butterflies + {conv / 1e6:.1f} M (conversion, as Shoup "
                                  f"products) + {final / 1e6:.1f} M final products"),
                    "algorithmic_bytes": 8 * N * (L + K + L) * 8}

    def e2e_step(self):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.step()
        self.o_pin.copy_(self.out, non_blocking=True)
        return self.x_pin.numel() * 8, self.o_pin.numel() * 8

    def oracle_setup(self):
        import oracle
        from ntt_arithmetic_gb300 import inputs
        self.o_qp = [int(v) for v in oracle.primes(2 * N, L + K)]
        self.o_ps = oracle.psis(self.o_qp, N)
        self.o_x = inputs.uniform_residues((2, L + K, N), self.o_qp, 31, buffer=7)

    def oracle_sample(self):
        import oracle
        t0 = time.perf_counter()
        oracle.moddown_ntt_batch(self.o_x, self.o_qp, self.o_ps, L, K, True)
        return time.perf_counter() - t0, 2, "2 of the 8 polynomials (INTT over QP, ModDown, NTT over Q)"


class HoistedRow(RowBench):
    name = "hoisted"
    metric = "hoisted rotations (key switches)/s, n=2^16, 24+8 primes, dnum=3, 16 Galois elements"
    unit = "key switch/s"
    R = 16
    workload = ("16 hoisted rotations k = 5^(2^r) mod 2n (r < 16) of one ciphertext component [1][24][n]: one "
                "ModUp + NTT of the 3 digits, then per rotation the automorphism fused into the inner product with "
                "that rotation's keys [16][3][2][32][n]; n=2^16")
    units_per_step = 16
    traffic_rows = 16 * 2 * (L + K)

    def setup(self, dev):
        import torch
        from ntt_arithmetic_gb300 import api
        q = api.find_primes(LOG_N, L)
        self.qp = q + api.find_primes(LOG_N, K, below=q[-1])
        self.t = api.NttTables(LOG_N, self.qp, dev)
        self.mt = api.ModupTables(L, K, DNUM, self.qp, dev)
        self.ks = [pow(5, 1 << r, 2 * N) for r in range(self.R)]
        self.x = _rand_dev((1,), q, N, 41, dev)
        self.keys = _rand_dev((self.R, DNUM, 2), self.qp, N, 42, dev)
        self.out = torch.empty((self.R, 1, 2, L + K, N), dtype=torch.uint64, device=dev)
        self.ws = torch.empty(api.keyswitch_workspace_bytes(LOG_N, L, K, DNUM, 1) // 8, dtype=torch.uint64,
                              device=dev)
        self.digits = self.ws.view(1, DNUM, L + K, N)
        self.x_pin = self.x.cpu().pin_memory()
        self.o_pin = torch.empty(self.out.shape, dtype=torch.uint64).pin_memory()

    def step(self):
        from ntt_arithmetic_gb300 import api
        api.keyswitch_hoisted(self.out, self.x, self.keys, self.ks, L, K, DNUM, self.t, self.mt, self.ws)

    def separate_ms(self, reps):
        from ntt_arithmetic_gb300 import api

        def fn():
            for r in range(self.R):
                api.keyswitch_ip(self.out[r], self.x, self.keys[r], L, K, DNUM, self.t, self.mt, self.ws)
        return _time_calls(fn, reps)

    def probe(self):
        from ntt_arithmetic_gb300 import api
        api.keyswitch_decompose(self.digits, self.x, L, K, DNUM, self.t, self.mt)
        plane = (L + K) * N * 8
        bytes_ = self.R * DNUM * 2 * plane + self.R * 2 * plane + DNUM * plane
        fn = lambda: api.keyswitch_apply(self.out, self.digits, self.keys, L, K, DNUM, self.t, galois=self.ks)
        return fn, {"bound": "hbm", "work": bytes_, "unit": "GB/s",
                    "kernel": "k_ks_ip_aut (automorphism fused into the key-switch inner product, 16 rotations)",
                    "work_note": "keys 16x3x2x32xn + outputs 16x2x32xn + digits 3x32xn words, 8 B each"}

    def e2e_step(self):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.step()
        self.o_pin.copy_(self.out, non_blocking=True)
        return self.x_pin.numel() * 8, self.o_pin.numel() * 8

    def oracle_setup(self):
        import oracle
        from ntt_arithmetic_gb300 import inputs
        self.o_qp = [int(v) for v in oracle.primes(2 * N, L + K)]
        self.o_ps = oracle.psis(self.o_qp, N)
        self.o_x = inputs.uniform_residues((1, L, N), self.o_qp[:L], 41, buffer=7)
        self.o_keys = inputs.uniform_residues((4, DNUM, 2, L + K, N), self.o_qp, 42, buffer=7)

    def oracle_sample(self):
        import oracle
        ks = [pow(5, 1 << r, 2 * N) for r in range(4)]
        t0 = time.perf_counter()
        oracle.keyswitch_hoisted_batch(self.o_x, self.o_keys, ks, self.o_qp, self.o_ps, L, K, DNUM)
        return time.perf_counter() - t0, 4, "4 of the 16 rotations (one ModUp + NTT of the digits, 4 x automorphism + IP)"


CHAIN_LOG_N, CHAIN_L = 11, 2100


class ModraiseRow(RowBench):
    name = "modraise"
    metric = "modraise polys/s, n=2^11, level-0 -> 2100-prime chain"
    unit = "poly/s"
    workload = ("modraise (exact Garner extension) of 4 level-0 ciphertexts [4][2][1][n] to the 2100-prime boot "
                "chain [4][2][2100][n], n=2^11; also timed: the exact and approximate conversion of one 8-prime "
                "key-switch digit to 32 primes at n=2^16")
    units_per_step = 8
    traffic_rows = 8 * CHAIN_L

    def setup(self, dev):
        import torch
        from ntt_arithmetic_gb300 import api
        self.chain = api.find_primes(CHAIN_LOG_N, CHAIN_L)
        n = 1 << CHAIN_LOG_N
        self.bt = api.BconvTables(self.chain[:1], self.chain, dev)
        self.x = _rand_dev((8,), self.chain[:1], n, 51, dev)
        self.out = torch.empty((8, CHAIN_L, n), dtype=torch.uint64, device=dev)
        self.x_pin = self.x.cpu().pin_memory()
        self.o_pin = torch.empty(self.out.shape, dtype=torch.uint64).pin_memory()
        q = api.find_primes(LOG_N, L)
        qp = q + api.find_primes(LOG_N, K, below=q[-1])
        self.dt = api.BconvTables(qp[:8], qp, dev)
        self.dx = _rand_dev((4,), qp[:8], N, 52, dev)
        self.dout = torch.empty((4, L + K, N), dtype=torch.uint64, device=dev)

    def step(self):
        from ntt_arithmetic_gb300 import api
        api.modraise(self.out, self.x, self.bt)

    def extra(self, reps):
        from ntt_arithmetic_gb300 import api
        ex = _time_calls(lambda: api.bconv(self.dout, self.dx, self.dt), reps)
        ap = _time_calls(lambda: api.bconv(self.dout, self.dx, self.dt, approx=True), reps)
        return {"digit_bconv_8_to_32_n65536_batch4_ms": {"exact": ex, "approx": ap}}

    def probe(self):
        from ntt_arithmetic_gb300 import api
        n = 1 << CHAIN_LOG_N
        bytes_ = 8 * n * 8 + 8 * CHAIN_L * n * 8
        fn = lambda: api.modraise(self.out, self.x, self.bt)
        return fn, {"bound": "hbm", "work": bytes_, "unit": "GB/s",
                    "kernel": "k_bconv<1,exact> (modraise, 8 polys, 1 -> 2100 primes)",
                    "work_note": "8 input limbs + 8 x 2100 output limbs of 2^11 words"}

    def e2e_step(self):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.step()
        self.o_pin.copy_(self.out, non_blocking=True)
        return self.x_pin.numel() * 8, self.o_pin.numel() * 8

    def oracle_setup(self):
        import oracle
        from ntt_arithmetic_gb300 import inputs
        self.o_chain = [int(v) for v in oracle.primes(2 << CHAIN_LOG_N, CHAIN_L)]
        self.o_x = inputs.uniform_residues((8, 1, 1 << CHAIN_LOG_N), self.o_chain[:1], 51, buffer=7)

    def oracle_sample(self):
        import oracle
        t0 = time.perf_counter()
        oracle.bconv_batch(self.o_x, self.o_chain[:1], self.o_chain)
        return time.perf_counter() - t0, 8, "all 8 polynomials (1 -> 2100 primes)"


class ChainRow(RowBench):
    name = "chain2100"
    CL = CHAIN_L
    metric = "NTT (poly x prime)/s on the 2100-prime chain, n=2^11"
    unit = "NTT (poly x prime)/s"
    workload = ("n=2^11, 2100-prime boot chain: fwd NTT of 16 polys (4 ciphertext pairs) -> tensor -> inv NTT of "
                "the 12 product polys")
    units_per_step = 28 * CHAIN_L
    traffic_rows = 16 * CHAIN_L

    def setup(self, dev):
        import torch
        from ntt_arithmetic_gb300 import api, inputs
        self.chain = api.find_primes(CHAIN_LOG_N, self.CL)
        n = 1 << CHAIN_LOG_N
        self.t = api.NttTables(CHAIN_LOG_N, self.chain, dev)
        host = inputs.uniform_residues((2, PAIRS, 2, self.CL, n), self.chain, 61, buffer=0)
        self.x_pin = torch.from_numpy(host).pin_memory()
        self.X = self.x_pin.to(dev)
        self.D = torch.empty((PAIRS, 3, self.CL, n), dtype=torch.uint64, device=dev)
        self.o_pin = torch.empty(self.D.shape, dtype=torch.uint64).pin_memory()

    def step(self):
        from ntt_arithmetic_gb300 import api
        api.ntt_fwd(self.X, self.t)
        api.tensor(self.D, self.X[0], self.X[1], self.t)
        api.ntt_inv(self.D, self.t)

    def probe(self):
        from ntt_arithmetic_gb300 import api
        n = 1 << CHAIN_LOG_N
        bfly = 16 * self.CL * (n // 2) * CHAIN_LOG_N
        fn = lambda: api.ntt_fwd(self.X, self.t)
        return fn, {"bound": "alu", "work": bfly, "peak": ALU_PEAK_BFLY / 1e9, "unit": "Gbutterfly/s",
                    "kernel": f"k_ntt_fwd<11,0,7,4,4> (16 polys x {self.CL} primes)",
                    "work_note": f"16 x {self.CL} transforms x 1024 x 11 butterflies",
                    "algorithmic_bytes": 16 * 16 * self.CL * n}

    def e2e_step(self):
        self.X.copy_(self.x_pin, non_blocking=True)
        self.step()
        self.o_pin.copy_(self.D, non_blocking=True)
        return self.x_pin.numel() * 8, self.o_pin.numel() * 8


    def oracle_setup(self):
        import oracle
        from ntt_arithmetic_gb300 import inputs
        chain = [int(v) for v in oracle.primes(2 << CHAIN_LOG_N, self.CL)]
        self.o_qs = chain[:self.CL]
        self.o_ps = oracle.psis(self.o_qs, 1 << CHAIN_LOG_N)
        self.o_x = inputs.uniform_residues((2, 1, 2, self.CL, 1 << CHAIN_LOG_N), self.o_qs, 61, buffer=7)

    def oracle_sample(self):
        import oracle
        threads = oracle.default_threads()
        t0 = time.perf_counter()
        X = oracle.ntt_batch(self.o_x, self.o_qs, self.o_ps, threads=threads)
        D = oracle.tensor_batch(X[0], X[1], self.o_qs)
        oracle.ntt_batch(D, self.o_qs, self.o_ps, inverse=True, threads=threads)
        return (time.perf_counter() - t0, 7 * self.CL,
                f"1 of the 4 ciphertext pairs on all {self.CL} primes, {threads} threads")


class LayerRow(ChainRow):
    name = "layer112"
    CL = 112
    metric = "NTT (poly x prime)/s on the 112-prime layer chain, n=2^11"
    workload = ("n=2^11, 112-prime layer chain (4 token positions x 2 components = 4 ciphertext pairs, 3.5 MiB per "
                "ciphertext): fwd NTT of 16 polys -> tensor -> inv NTT of the 12 product polys")
    units_per_step = 28 * 112
    traffic_rows = 16 * 112
    l2 = ("inputs 29 MB (< L2): a 256 MB write flushes L2 before every step, outside the timed region (each step "
          "is bracketed by its own events and the step times are summed)")

    def setup(self, dev):
        import torch
        super().setup(dev)
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def before_step(self):
        self.flush.zero_()


class Pr1Row(RowBench):
    """The small parity configuration: n = 2^11, the 4 largest primes q < 2^50
    with q = 1 mod 2^12, one pair of polynomials a, b: forward NTT of both,
    pointwise product, inverse NTT (the negacyclic product a*b).  It is
    launch- and latency-bound (64 KB per polynomial); reported, not graded."""
    name = "pr1"
    metric = "NTT (poly x prime)/s, negacyclic product at n=2^11, 4 primes"
    unit = "NTT (poly x prime)/s"
    workload = ("n=2^11, L=4 (the 4 largest q<2^50, q=1 mod 4096), 1 pair of polynomials: fwd NTT of both -> "
                "pointwise product -> inv NTT (the negacyclic product)")
    units_per_step = 12                       # 8 forward + 4 inverse transforms
    traffic_rows = 8
    l2 = ("inputs 128 KB (< L2): a 256 MB write flushes L2 before every step, outside the timed region (each step "
          "is bracketed by its own events and the step times are summed)")
    LOG_N, L = 11, 4

    def setup(self, dev):
        import torch
        from ntt_arithmetic_gb300 import api, inputs
        n = 1 << self.LOG_N
        self.q = api.find_primes(self.LOG_N, self.L)
        self.t = api.NttTables(self.LOG_N, self.q, dev)
        host = np.concatenate([inputs.uniform_residues((1, self.L, n), self.q, 1, buffer=b) for b in (0, 1)])
        self.x_pin = torch.from_numpy(host).pin_memory()
        self.X = self.x_pin.to(dev)
        self.P = torch.empty((self.L, n), dtype=torch.uint64, device=dev)
        self.o_pin = torch.empty(self.P.shape, dtype=torch.uint64).pin_memory()
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.graph = None
        self.graph = self.capture()
        self.X.copy_(self.x_pin)                  # the warm-up before the capture transformed X

    def capture(self):
        """Capture the step's three launches once in a CUDA graph: at this size
        one ctypes call costs more host time than its kernel takes on the GPU."""
        import torch
        from ntt_arithmetic_gb300 import api
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.eager_step()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        c0 = api.launch_count()
        with torch.cuda.graph(g):
            self.eager_step()
        self.graph_launches = api.launch_count() - c0
        return g

    def before_step(self):
        self.flush.zero_()

    def eager_step(self):
        from ntt_arithmetic_gb300 import api
        api.ntt_fwd(self.X, self.t)
        api.mul_ntt(self.P, self.X[0], self.X[1], self.t)
        api.ntt_inv(self.P, self.t)

    def step(self):
        if self.graph is None:
            self.eager_step()
        else:
            self.graph.replay()

    def replayed_launches(self, steps):
        return self.graph_launches * steps if self.graph is not None else 0

    def extra(self, reps):
        return {"eager_ms_per_step": _time_calls(self.eager_step, reps),
                "launch": "timed steps replay a CUDA graph of the step's 3 kernels, captured once; "
                          "eager_ms_per_step issues them as 3 API calls, back to back, without the L2 flush"}

    def probe(self):
        from ntt_arithmetic_gb300 import api
        import torch
        n = 1 << self.LOG_N
        reps = 32                                 # launches per replay: the host cost of one call exceeds the kernel's
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                api.ntt_fwd(self.X, self.t)
        return g.replay, {
            "bound": "alu", "work": 2 * self.L * (n // 2) * self.LOG_N, "launches_per_call": reps,
            "peak": ALU_PEAK_BFLY / 1e9, "unit": "Gbutterfly/s",
            "kernel": "k_ntt_fwd<11,0,7,4,4> (2 polys x 4 primes: 8 CTAs), timed as 32 launches in one CUDA graph",
            "work_note": "8 transforms x 1024 x 11 butterflies; 8 CTAs on 152 SMs: launch- and latency-bound, the "
                         "ALU fraction is reported, not a target",
            "algorithmic_bytes": 16 * 2 * self.L * n}

    def e2e_step(self):
        self.X.copy_(self.x_pin, non_blocking=True)
        self.eager_step()
        self.o_pin.copy_(self.P, non_blocking=True)
        return self.x_pin.numel() * 8, self.o_pin.numel() * 8

    def oracle_setup(self):
        import oracle
        from ntt_arithmetic_gb300 import inputs
        self.o_q = [int(v) for v in oracle.primes(2 << self.LOG_N, self.L)]
        self.o_ps = oracle.psis(self.o_q, 1 << self.LOG_N)
        self.o_x = np.concatenate([inputs.uniform_residues((1, self.L, 1 << self.LOG_N), self.o_q, 1, buffer=b)
                                   for b in (0, 1)])

    def oracle_sample(self):
        import oracle
        threads = oracle.default_threads()
        t0 = time.perf_counter()
        reps = 200
        for _ in range(reps):
            X = oracle.ntt_batch(self.o_x, self.o_q, self.o_ps, threads=threads)
            Pr = oracle.mul_batch(X[0:1], X[1:2], self.o_q)
            oracle.ntt_batch(Pr, self.o_q, self.o_ps, inverse=True, threads=threads)
        return (time.perf_counter() - t0, 12 * reps, f"the whole step, {reps} times, {threads} threads")


ROWS = {r.name: r for r in (ModdownRow, HoistedRow, ModraiseRow, ChainRow, LayerRow, Pr1Row)}


def row_bench(args):
    import torch
    from ntt_arithmetic_gb300 import api
    from ntt_arithmetic_gb300 import build as B
    ws, rank, local = dist_env()
    row = ROWS[args.workload]()
    if args.impl == "reference":
        if rank != 0:
            return
        from oracle import build as OB
        OB.build() if OB.stale() else None
        import oracle
        row.oracle_setup()
        for _ in range(min(args.warmup, 1)):
            row.oracle_sample()
        samples = [row.oracle_sample() for _ in range(args.steps)]
        dt = sum(s[0] for s in samples)
        units = sum(s[1] for s in samples)
        value = units / dt
        print(json.dumps({
            "impl": "reference", "metric": row.metric, "value": value, "unit": row.unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u64",
            "data": "synthetic: seeded uniform residues in [0, q)", "config": row.config(),
            "cpu_baseline": {"value": value, "unit": row.unit, "cores": oracle.default_threads(), "kind": "oracle",
                             "sample": samples[0][2]},
            "e2e": {"value": value, "unit": row.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    import torch.distributed as dist
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(B.OUT):
        B.build()
    if ws > 1:
        dist.barrier()
    row.setup(dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        row.before_step()
        row.step()
    barrier()
    launches0 = api.launch_count()
    evs = _events(2 * args.steps)
    with ClockSampler(local) as clk:
        barrier()
        poll = NvmlClockPoller(dev).start()
        for i in range(args.steps):
            row.before_step()
            evs[2 * i].record(stream)
            row.step()
            evs[2 * i + 1].record(stream)
        barrier()
        poll.stop()
    launches = api.launch_count() - launches0 + row.replayed_launches(args.steps)
    ms = max_over_ranks(sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(args.steps)) / args.steps, dev)
    fn, roof = row.probe()
    kms = _time_calls(fn, max(3, args.steps)) / roof.pop("launches_per_call", 1)
    achieved = roof.pop("work") / (kms * 1e-3) / 1e9
    hbm, hbm_kind = peaks()
    if roof["bound"] == "hbm":
        roof["peak"], roof["peak_kind"] = hbm, hbm_kind
    else:
        roof["peak_kind"] = "derived: measured integer-pipe rates x 152 SMs x 2070 MHz"
    roof.update({"achieved": achieved, "frac": achieved / roof["peak"], "kernel_ms": kms,
                 "traffic": kernel_traffic(row.name, row.traffic_rows), "traffic_unit": "bytes/launch",
                 "traffic_source": TRAFFIC_SOURCE})
    barrier()
    n_e2e = max(1, min(args.steps, 5))
    for _ in range(max(2, args.warmup)):   # untimed: the first copies through the pinned buffers
        row.e2e_step()
    barrier()
    f0, f1 = _events(2)
    f0.record(stream)
    for _ in range(n_e2e):
        h2d, d2h = row.e2e_step()
    f1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / n_e2e, dev)
    line = {
        "metric": row.metric, "value": whole_job_rate(row.units_per_step, ws, ms), "unit": row.unit,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u64",
        "data": "synthetic: seeded uniform residues in [0, q) (SplitMix64 counter generator)",
        "config": dict(row.config(), parallelism=f"replicas x{ws}"),
        "roofline": roof, "clocks": clock_record(poll, clk), "gpu_launches": launches,
        "e2e": {"value": whole_job_rate(row.units_per_step, ws, e2e_ms), "unit": row.unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
    }
    if isinstance(row, HoistedRow):
        sep = row.separate_ms(max(3, args.steps // 2))
        line["separate_keyswitch_ms_per_step"] = sep
        line["hoisting_speedup"] = sep / ms
    if isinstance(row, (ModraiseRow, Pr1Row)):
        line.update(row.extra(max(3, args.steps)))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        from oracle import build as OB
        OB.build() if OB.stale() else None
        row.oracle_setup()
        dt, units, desc = row.oracle_sample()
        line["cpu_baseline"] = {"value": units / dt, "unit": row.unit, "cores": oracle.default_threads(),
                                "kind": "oracle", "sample": f"{desc}; {dt:.2f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-steps", type=int, default=2)
    ap.add_argument("--sweep", action="store_true", help="time every point of the n / L / batch sweep instead")
    ap.add_argument("--sweep-reps", type=int, default=5)
    ap.add_argument("--workload", choices=["step"] + sorted(ROWS), default="step",
                    help="step: the headline hot-path step; the others time one widened row each")
    args = ap.parse_args()
    if args.workload != "step":
        row_bench(args)
    elif args.sweep:
        sweep(args)
    elif args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
