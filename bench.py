#!/usr/bin/env python
"""Benchmark of the DMS decode hot path on B300.

One step = one pass of the whole hot path for one token of every sequence:
the fused append/evict kernel (decision, delayed eviction, slot reuse, K/V
write) and the split-K decode-attention kernel over the compacted caches
(whose last-arriving warps merge the partial results of heads split across
warps).  Workload (default): Qwen3-8B-like attention -- batch 32, 32 query /
8 KV heads, head_dim 128, window 16, eviction logits N(1.150, 1) (CR 8) --
timed at context ~16K: the cache is filled to 16384 - W - 2K tokens with
chunked appends, then W warm-up steps, K timed steps (pass A) and K steps with
per-call events (pass B) end at 16384; pass C repeats the last decode call K
times back to back.  The retained K/V (~270 MB) is larger than the 126 MB L2,
so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Prints one JSON line on rank 0.  ``--impl reference`` times the CPU oracle on
the host cores (the reference arm); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn tokens/s and achieved HBM GB/s (% of peak) at CR 8, Qwen3-8B shapes"
SETTLE_CALLS = 256  # untimed read-only decode calls before a timed leg's warm-up
NOMINAL_HBM_GBS = 8000.0  # "roughly 8 TB/s" stated with the target
FALLBACK_HBM_GBS = 6400.0
PROFILE_FILE = os.path.join(ROOT, "profiles", "decode_kernel_fused_step_qwen3-8b_cr8_n16384.md")
KERNEL_SOURCES = ["decode.cuh", "dms_device.cuh"]


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def code_only(text: str) -> str:
    """C/C++ source without its comments and blank lines, so that the stamp on
    a profile follows the code and survives edits of comments alone."""
    out, i, n = [], 0, len(text)
    quote = None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 1
            elif c == quote:
                quote = None
        elif c in "\"'":
            quote = c
            out.append(c)
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            continue
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            continue
        else:
            out.append(c)
        i += 1
    lines = (ln.rstrip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    """Stamp of the decode kernel's code (comments and blank lines excluded)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "learned_kv_cache_eviction_b300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    try:
        text = open(PROFILE_FILE).read()
    except OSError:
        return None
    vals = {}
    for ln in text.splitlines():
        t = ln.strip().lstrip("-* ").strip()
        if t.startswith(("traffic_bytes_per_launch", "kernel_source_sha256")) and ":" in t:
            k, v = t.split(":", 1)
            v = v.strip()
            if v.startswith("`"):  # the value in backticks, then an optional note
                v = v[1:].split("`", 1)[0]
            vals[k.strip()] = v.split()[0] if v else v
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# A spin kernel of about a millisecond (torch.cuda._sleep) queued ahead of a
# device-timed region's start event, so that all of the region's launches are
# enqueued before the GPU reaches them: the region then times the device
# running them back to back, not the host's launch latency and scheduling
# jitter at its start (without it, 20-step regions on one box measured 57-74 µs
# per step for 55 µs steps).  The end-to-end leg, which is meant to include the
# host, is not gated.  The start event is a timing event, which ends the
# programmatic early start, so no part of a timed step runs before it.
GATE_CYCLES = 2_000_000


def gate() -> None:
    torch.cuda._sleep(GATE_CYCLES)


class _Nvml:
    """Minimal read-only NVML access through ctypes (clock and clock-event
    reason queries only; nothing is set)."""

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")

    def handle_from(self, pci: str, device_index: int):
        """The NVML handle of the GPU at PCI address `pci` (as CUDA reports it),
        else of NVML index `device_index`."""
        ct = self.ct
        h = ct.c_void_p()
        if pci and self.lib.nvmlDeviceGetHandleByPciBusId_v2(ct.c_char_p(pci.encode()), ct.byref(h)) == 0:
            return h
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(device_index), ct.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return h

    def sm_clock(self, h) -> int:
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(h, 1, self.ct.byref(v))  # NVML_CLOCK_SM
        return int(v.value)

    def sm_max_clock(self, h) -> int:
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(h, 1, self.ct.byref(v))
        return int(v.value)

    def reasons(self, h) -> int:
        v = self.ct.c_ulonglong()
        self.lib.nvmlDeviceGetCurrentClocksEventReasons(h, self.ct.byref(v))
        return int(v.value)


def _clock_poll(conn, pci: str, device_index: int) -> None:
    """Clock sampler process (spawned; no CUDA): on each "sample" message from
    the parent it reads the SM clock and the clock-event reasons through NVML
    (read-only), stamped with time.monotonic(); on "stop" it sends the samples
    back and exits."""
    try:
        nv = _Nvml()
        h = nv.handle_from(pci, device_index)
        conn.send(("ok", nv.sm_max_clock(h)))
    except Exception as exc:
        conn.send(("err", repr(exc)[:200]))
        return
    samples = []
    while True:
        msg = conn.recv()
        if msg == "stop":
            conn.send(samples)
            return
        try:
            samples.append((time.monotonic(), nv.sm_clock(h), nv.reasons(h)))
        except Exception:
            pass


class ClockSampler:
    """Reads the SM clock and clock-event reasons through NVML (read-only)
    while the timed steps run on the GPU.  The reads are made by a process of
    its own, on request (`sample()`, called after enqueueing some of the timed
    steps, so that the GPU is still running them), so that they neither hold
    this process's interpreter lock while steps are being enqueued nor poll
    the GPU all the time (continuous NVML polling, even every 2 ms, slowed the
    timed steps by a few per cent)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting"}

    def __init__(self, device_index: int):
        import multiprocessing as mp
        self.ok = False
        self.err = ""
        self.samples, self.reasons = [], set()
        self.t0 = self.t1 = None
        try:
            p = torch.cuda.get_device_properties(device_index)
            pci = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except Exception:
            pci = ""
        ctx = mp.get_context("spawn")
        self.conn, child = ctx.Pipe()
        self.proc = ctx.Process(target=_clock_poll, args=(child, pci, device_index), daemon=True)
        self.proc.start()

    def _ready(self):
        if self.ok or self.err:
            return
        try:
            if not self.conn.poll(120):
                raise RuntimeError("clock sampler did not start")
            tag, val = self.conn.recv()
        except Exception as exc:
            tag, val = "err", repr(exc)[:200]
        if tag == "ok":
            self.ok, self.max_mhz = True, val
        else:
            self.err = val

    def sample(self):
        """Ask for one reading now (does not wait for it)."""
        if self.ok:
            self.conn.send("sample")

    def __enter__(self):
        self._ready()
        self.t0 = time.monotonic()
        return self

    def __exit__(self, *a):
        self.t1 = time.monotonic()
        if self.ok:
            self.conn.send("stop")
            got = self.conn.recv()
            self.samples = [x[1] for x in got]
            self.stamps_inside = sum(1 for x in got if self.t0 <= x[0] <= self.t1)
            for _, _, r in got:
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
        self.proc.join(timeout=10)
        return False

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": f"NVML unavailable: {self.err}"}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "samples_inside_timed_region": self.stamps_inside,
                "source": "NVML (ctypes), read by a separate process on request while the GPU runs the timed "
                          "steps (after half of them and after all of them were enqueued)"}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


# ---------------------------------------------------------------------------
# the native arm
# ---------------------------------------------------------------------------

def fill_cache(dms, W, wl, n0, device, layer=0, kv_format="bf16"):
    cache = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, device=device, kv_format=kv_format)
    t = 0
    while t < n0:
        n = min(512, n0 - t)
        k, v, lg = W.kv_range(wl, layer, t, t + n, device=device)
        cache.append_chunk(k, v, lg)
        t += n
    torch.cuda.synchronize(device)
    return cache


def step_inputs(W, wl, t0, n, device, layer=0):
    k, v, lg = W.kv_range(wl, layer, t0, t0 + n, device=device)
    q = W.q_range(wl, layer, t0, t0 + n, device=device)
    return ([q[:, :, i].contiguous() for i in range(n)], [k[:, :, i].contiguous() for i in range(n)],
            [v[:, :, i].contiguous() for i in range(n)], [lg[:, :, i].contiguous() for i in range(n)])


def time_device_leg(dms, cache, ins, warmup, steps, scale, device, clocks=None, dist=None):
    """Warm-up, then three passes through the C ABI on device-resident inputs.
    Pass A (the headline): ``steps`` calls of dms_step (append + decode in one
    launch of the fused decode kernel), events only around the whole pass, so
    consecutive launches keep their programmatic-launch overlap; the pass's
    mean is that kernel's in-stream duration.  Pass B: ``steps`` more steps as
    dms_append + dms_decode_attention with events around every decode call;
    the events break the launch overlap, so these per-call times carry a
    launch gap each.  Pass C: ``steps`` back-to-back dms_decode_attention
    calls on the final cache state, events around the whole pass -- the plain
    decode kernel's average in-stream duration.  The retained K/V (> 126 MB
    L2) is re-read from HBM by every call.  Passes A and C start behind a
    gate() kernel, so that they time the device, not the host's launches."""
    lib = dms.load_library()
    h = cache.handle
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    qs, ks, vs, ls = ins
    Hq = qs[0].shape[1]
    out = torch.empty((cache.batch, Hq, cache.head_dim), dtype=torch.float32, device=device)
    outp = out.data_ptr()

    def append(i):
        rc = lib.dms_append(h, ks[i].data_ptr(), vs[i].data_ptr(), ls[i].data_ptr(), sh)
        if rc:
            raise dms.DmsError(rc, "dms_append")

    def decode(i):
        rc = lib.dms_decode_attention(h, qs[i].data_ptr(), outp, scale, Hq, sh)
        if rc:
            raise dms.DmsError(rc, "dms_decode_attention")

    def step(i):
        rc = lib.dms_step(h, ks[i].data_ptr(), vs[i].data_ptr(), ls[i].data_ptr(), qs[i].data_ptr(), outp, scale,
                          Hq, sh)
        if rc:
            raise dms.DmsError(rc, "dms_step")

    # Untimed settling before the warm-up steps: read-only decode calls on the
    # filled cache (no state changes) for a few ms, so that the timed steps do
    # not see the GPU's ramp from idle after the fill (a fresh box once ran the
    # first ~15 ms of kernels 3-4x slower).
    for _ in range(SETTLE_CALLS):
        decode(0)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(device)
    len0 = int(cache.lengths().sum())
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    with (clocks if clocks is not None else _Null()):
        gate()
        t_start.record(stream)
        for i in range(warmup, warmup + steps):
            step(i)
            if clocks is not None and i in (warmup + steps // 2, warmup + steps - 1):
                clocks.sample()  # the GPU is still running the steps enqueued so far
        t_stop.record(stream)
        torch.cuda.synchronize(device)
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_stop)
    len1 = int(cache.lengths().sum())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for j in range(steps):
        i = warmup + steps + j
        eva[j][0].record(stream)
        append(i)
        eva[j][1].record(stream)
        ev[j][0].record(stream)
        decode(i)
        ev[j][1].record(stream)
    torch.cuda.synchronize(device)
    len2 = int(cache.lengths().sum())
    dec = [a.elapsed_time(b) * 1e3 for a, b in ev]
    app = [a.elapsed_time(b) * 1e3 for a, b in eva]
    last = warmup + 2 * steps - 1
    c_start = torch.cuda.Event(enable_timing=True)
    c_stop = torch.cuda.Event(enable_timing=True)
    gate()
    c_start.record(stream)
    for _ in range(steps):
        decode(last)
    c_stop.record(stream)
    torch.cuda.synchronize(device)
    st = cache.status()
    if st != dms.DMS_OK:
        raise dms.DmsError(st, "device status after the timed steps")
    return {"total_ms": total_ms, "decode_us_call": statistics.mean(dec), "append_us_call": statistics.mean(app),
            "decode_us_call_median": statistics.median(dec),
            "decode_us": c_start.elapsed_time(c_stop) * 1e3 / steps,
            "len_sum_start": len0, "len_sum_end": len1, "len_sum_b": 0.5 * (len1 + len2), "len_sum_c": len2}


def time_e2e_leg(dms, W, wl, n0, warmup, steps, device, dist=None):
    """The same steps through the public API with host buffers: every step's
    inputs (k, v, logits, q) sit in pinned host memory and its output is read
    back into pinned host memory, by DmsCache.step_host -> dms_step_host.  The
    library copies each step's rows in on its own copy stream, runs the fused
    step on the compute stream and copies the output out on a second copy
    stream, with two sets of device rows so that step i's copies overlap the
    steps i - 1 and i + 1.  The host enqueues ahead; the timed region ends
    when the last output is in host memory (host_join, then an event on the
    compute stream).  Every step has its own input and output buffers;
    each is copied from or to once before the timed region, as a serving
    loop's reused buffers would have been (a first copy out of or into freshly
    pinned pages costs several times a later one).
    Returns (ms for `steps` steps, input bytes per step, output bytes per step)."""
    cache = fill_cache(dms, W, wl, n0, device)
    ins = step_inputs(W, wl, n0, warmup + steps, device)
    n = warmup + steps
    qh, kh, vh, lh = ([x[i].contiguous().cpu().pin_memory() for i in range(n)] for x in ins)
    del ins
    in_bytes = sum(t[0].numel() * t[0].element_size() for t in (qh, kh, vh, lh))
    out_d = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device=device)
    out_h = torch.empty((n, wl.B, wl.Hq, wl.D), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(device)
    # Every pinned buffer is read or written by a copy once before the timed
    # region, as a serving loop's reused buffers would have been (a copy's
    # first touch of freshly pinned pages costs several times a later one).
    scratch = [torch.empty_like(t, device=device) for t in (qh[0], kh[0], vh[0], lh[0])]
    for i in range(n):
        out_h[i].copy_(out_d, non_blocking=True)
        for d, hsrc in zip(scratch, (qh[i], kh[i], vh[i], lh[i])):
            d.copy_(hsrc, non_blocking=True)
    torch.cuda.synchronize(device)
    del scratch

    def step(i):
        cache.step_host(kh[i], vh[i], lh[i], qh[i], out_h[i], wl.scale)

    # untimed settling after the fill, as in time_device_leg (read-only decodes)
    q_d = qh[0].to(device)
    for _ in range(SETTLE_CALLS):
        cache.decode_attention(q_d, out=out_d, scale=wl.scale)
    for i in range(warmup):
        step(i)
    cache.host_join()
    torch.cuda.synchronize(device)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(warmup, n):
        step(i)
    cache.host_join()
    t1.record(stream)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1)
    assert bool(torch.isfinite(out_h[warmup:]).all())
    cache.close()
    return ms, in_bytes, out_h[0].numel() * out_h.element_size()


def replica_workload(wl, rank: int):
    """Weak scaling: every rank serves its own batch of independent sequences,
    drawn with its own seed (rank 0 keeps the workload's seed)."""
    return wl.with_(seed=wl.seed + 1000 * rank) if rank else wl


def max_over_ranks(dist, x: float, device) -> float:
    """The slowest rank's time (identity on one process)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(batch: int, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: the tokens of all ranks over the slowest rank's time."""
    return batch * steps * world / (ms * 1e-3)


def decode_bytes(wl, len_sum):
    """Algorithmic bytes of one decode call: retained K and V (bf16), q (bf16),
    out (fp32) and the lengths (int32)."""
    return len_sum * 2 * wl.D * 2 + wl.B * wl.Hq * wl.D * (2 + 4) + wl.B * wl.Hkv * 4


def append_bytes(wl):
    """Algorithmic bytes of appending one token to every head: the new K and V
    rows read and written (bf16), its logit (fp32), the new length (int32), the
    ring entries of t - w read and of t written (slot int32 + mark byte) and its
    slot-map entry (int32)."""
    return wl.B * wl.Hkv * (4 * wl.D * 2 + 4 + 4 + 2 * 5 + 4)


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 1) for p in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_timer(wl, n_ctx, rows):
    """Draw the oracle's inputs on the CPU for batch rows ``rows`` up to context
    n_ctx; return a function running the oracle's decode step at position t."""
    import oracle.dms_oracle as O
    from learned_kv_cache_eviction_b300 import workload as W

    k, v, lg = W.kv_range(wl, 0, 0, n_ctx, rows=rows)
    q = W.q_range(wl, 0, n_ctx - 256, n_ctx, rows=rows)
    k_np, v_np = k.float().numpy(), v.float().numpy()
    e = O.eviction_decisions(lg.numpy())
    q_np = q.float().numpy()

    def run(t):
        return O.decode_attention(q_np[:, :, t - (n_ctx - 256)], k_np, v_np, e, t, wl.w, wl.scale)
    return run


def cpu_baseline(wl, n_ctx, seconds=12.0, rows=(0, 1), one_core_seconds=4.0):
    """The oracle timed on the host's cores (its BLAS threads), then on one
    core for a shorter sample."""
    run = oracle_timer(wl, n_ctx, list(rows))

    def sample(limit):
        t0 = time.perf_counter()
        steps = 0
        while True:
            run(n_ctx - 1 - (steps % 256))
            steps += 1
            if time.perf_counter() - t0 >= limit:
                break
        return steps, time.perf_counter() - t0

    steps, dt = sample(seconds)
    line = {"value": len(rows) * steps / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"oracle decode step (mask + dense softmax attention) for batch rows {list(rows)} of "
                      f"{wl.B} at positions {n_ctx - min(steps, 256)}..{n_ctx - 1} ({steps} steps, {dt:.1f} s)"}
    one = one_core_sample(wl.name, n_ctx, list(rows), one_core_seconds)
    if one is not None:
        line["one_core"] = one
    return line


def one_core_sample(name, n_ctx, rows, seconds):
    """The oracle's decode step on one core: a child process whose BLAS and
    OpenMP pools are limited to one thread by its environment."""
    import subprocess
    code = (
        "import json, sys, time\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "from learned_kv_cache_eviction_b300 import workload as W\n"
        f"run = bench.oracle_timer(W.WORKLOADS[{name!r}], {n_ctx}, {rows!r})\n"
        "t0 = time.perf_counter(); n = 0\n"
        f"while time.perf_counter() - t0 < {seconds}:\n"
        f"    run({n_ctx} - 1 - (n % 256)); n += 1\n"
        "dt = time.perf_counter() - t0\n"
        f"print(json.dumps({{'value': {len(rows)} * n / dt, 'unit': 'tokens/s', 'cores': 1, "
        "'sample': f'same, one thread, {n} steps, {dt:.1f} s'}))\n")
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    try:
        res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=seconds + 240)
        return json.loads(res.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def time_variants(dms, W, device, steps):
    """The ablation variants (eager eviction, windows 64 and 256, drifting CR)
    at the headline shapes: each cache is filled to 16384 tokens, then `steps`
    back-to-back dms_decode_attention calls are timed with events around the
    pass.  Reported: time per launch, algorithmic GB/s and the realised CR."""
    lib = dms.load_library()
    stream = torch.cuda.current_stream(device)
    rows = []
    for name in ("qwen3-8b-eager", "qwen3-8b-w64", "qwen3-8b-w256", "qwen3-8b-drift"):
        wl = W.WORKLOADS[name]
        cache = fill_cache(dms, W, wl, wl.cap, device)
        q = W.q_range(wl, 0, wl.cap - 1, wl.cap, device=device)[:, :, 0].contiguous()
        out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device=device)
        for _ in range(3):
            lib.dms_decode_attention(cache.handle, q.data_ptr(), out.data_ptr(), wl.scale, wl.Hq, stream.cuda_stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gate()
        e0.record(stream)
        for _ in range(steps):
            rc = lib.dms_decode_attention(cache.handle, q.data_ptr(), out.data_ptr(), wl.scale, wl.Hq,
                                          stream.cuda_stream)
            if rc:
                raise dms.DmsError(rc, "dms_decode_attention")
        e1.record(stream)
        torch.cuda.synchronize(device)
        us = e0.elapsed_time(e1) * 1e3 / steps
        len_sum = int(cache.lengths().sum())
        st = cache.status()
        cache.close()
        if st != dms.DMS_OK:
            raise dms.DmsError(st, name)
        rows.append({"workload": name, "window": wl.w, "context": wl.cap, "us_per_launch": us,
                     "achieved_GBps": decode_bytes(wl, len_sum) / (us * 1e-6) / 1e9,
                     "realised_cr": wl.B * wl.Hkv * wl.cap / len_sum, "note": wl.note})
    return rows


WORKLOAD_ROWS = ("tiny", "llama-3.2-1b", "qwen3-8b", "qwen-r1-32b", "long-context")
# The benchmark plan's literal logit distributions, whose realised compression
# differs from the stated one (secondary rows).
LITERAL_ROWS = ("llama-3.2-1b-literal", "qwen3-8b-literal", "long-context-literal")


def time_workloads(dms, W, device, steps, names=WORKLOAD_ROWS):
    """Decode throughput on every configured workload at its own shapes: the
    cache (one layer) is filled to the workload's final context (minus the
    timed steps), then `steps` dms_step calls (append + decode, one fused
    launch) and `steps` back-to-back dms_decode_attention calls, events around
    each pass.  Reported per workload: tokens/s of the step, the decode
    kernel's time, its algorithmic GB/s and fraction of the measured copy
    bandwidth and of the nominal 8 TB/s, the realised compression and the
    tokens held in memory at the end (the method's "peak tokens in memory":
    the retained total only grows over these runs)."""
    lib = dms.load_library()
    stream = torch.cuda.current_stream(device)
    peak, _ = measured_hbm_peak()
    rows = []
    for name in names:
        wl = W.WORKLOADS[name]
        n_end = wl.cap if not name.startswith("llama-3.2-1b") else wl.prefill + wl.decode
        n_end = min(n_end, wl.cap)
        n0 = n_end - steps - 3
        cache = fill_cache(dms, W, wl, n0, device)
        qs, ks, vs, ls = step_inputs(W, wl, n0, steps + 3, device)
        out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device=device)

        def step(i):
            rc = lib.dms_step(cache.handle, ks[i].data_ptr(), vs[i].data_ptr(), ls[i].data_ptr(), qs[i].data_ptr(),
                              out.data_ptr(), wl.scale, wl.Hq, stream.cuda_stream)
            if rc:
                raise dms.DmsError(rc, f"dms_step ({name})")

        for i in range(3):
            step(i)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gate()
        e0.record(stream)
        for i in range(3, steps + 3):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        step_us = e0.elapsed_time(e1) * 1e3 / steps
        len_sum = int(cache.lengths().sum())
        def decode():
            rc = lib.dms_decode_attention(cache.handle, qs[-1].data_ptr(), out.data_ptr(), wl.scale, wl.Hq,
                                          stream.cuda_stream)
            if rc:
                raise dms.DmsError(rc, f"dms_decode_attention ({name})")

        for _ in range(8):
            decode()
        gate()
        e0.record(stream)
        for _ in range(steps):
            decode()
        e1.record(stream)
        torch.cuda.synchronize(device)
        dec_us = e0.elapsed_time(e1) * 1e3 / steps
        st = cache.status()
        cache.close()
        if st != dms.DMS_OK:
            raise dms.DmsError(st, name)
        gbs = decode_bytes(wl, len_sum) / (dec_us * 1e-6) / 1e9
        rows.append({"workload": name, "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D,
                     "context": n_end, "logits": list(wl.logits), "realised_cr": wl.B * wl.Hkv * n_end / len_sum,
                     "peak_tokens_in_memory": len_sum,
                     "step_tokens_per_s": wl.B / (step_us * 1e-6), "step_us": step_us,
                     "decode_us": dec_us, "decode_GBps": gbs, "decode_frac_of_measured_copy": gbs / peak,
                     "decode_frac_of_nominal_8TBps": gbs / NOMINAL_HBM_GBS})
        del qs, ks, vs, ls
        torch.cuda.empty_cache()
    return rows


def time_context_sweep(dms, W, device, names=("qwen3-8b", "qwen-r1-32b"), points=(1024, 2048, 4096, 8192, 16384),
                       reps=20):
    """Decode time of one layer at growing context: the cache is filled in
    chunks up to each point, then `reps` dms_decode_attention calls are timed
    one by one with events, each after a write of twice the L2 size (below
    16K the retained K/V fits in L2).  Reported per point: the median call,
    tokens/s, algorithmic GB/s and its fraction of the measured copy
    bandwidth."""
    lib = dms.load_library()
    stream = torch.cuda.current_stream(device)
    peak, _ = measured_hbm_peak()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    out_rows = []
    for name in names:
        wl = W.WORKLOADS[name]
        cache = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, device=device)
        out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device=device)
        t = 0
        for n in points:
            while t < n:
                m = min(512, n - t)
                k, v, lg = W.kv_range(wl, 0, t, t + m, device=device)
                cache.append_chunk(k, v, lg)
                t += m
            q = W.q_range(wl, 0, n - 1, n, device=device)[:, :, 0].contiguous()
            times = []
            for r in range(reps + 3):
                flush.sum()  # reads twice the L2 size: evicts the cache, leaves no dirty lines
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                rc = lib.dms_decode_attention(cache.handle, q.data_ptr(), out.data_ptr(), wl.scale, wl.Hq,
                                              stream.cuda_stream)
                e1.record(stream)
                if rc:
                    raise dms.DmsError(rc, f"dms_decode_attention ({name}, n={n})")
                torch.cuda.synchronize(device)
                if r >= 3:
                    times.append(e0.elapsed_time(e1) * 1e3)
            us = statistics.median(times)
            len_sum = int(cache.lengths().sum())
            gbs = decode_bytes(wl, len_sum) / (us * 1e-6) / 1e9
            out_rows.append({"workload": name, "context": n, "realised_cr": wl.B * wl.Hkv * n / len_sum,
                             "decode_us_median": us, "tokens_per_s": wl.B / (us * 1e-6), "decode_GBps": gbs,
                             "frac_of_measured_copy": gbs / peak})
        st = cache.status()
        cache.close()
        if st != dms.DMS_OK:
            raise dms.DmsError(st, f"context sweep ({name})")
    del flush
    return {"note": f"L2 flushed (a {2 * l2 >> 20} MB read) before every call; median of {reps} calls, "
                    "each timed alone with events (so each includes its launch gap)", "points": out_rows}


def decode_bytes_fp8(wl, len_sum):
    """Algorithmic bytes of one decode call on an FP8 cache: per retained slot
    the K row (D codes + its 16-byte scale chunk) and the V row (D codes); q,
    out and lengths as for bf16."""
    return len_sum * (2 * wl.D + 16) + wl.B * wl.Hq * wl.D * (2 + 4) + wl.B * wl.Hkv * 4


def time_fp8_leg(dms, W, wl, device, steps):
    """FP8 (E4M3) storage at the headline shapes: the cache is filled to
    16384 - steps tokens, then `steps` timed dms_step calls (append + decode,
    one fused launch, as for bf16 storage) and `steps` back-to-back
    dms_decode_attention calls, with events around each pass."""
    lib = dms.load_library()
    stream = torch.cuda.current_stream(device)
    n0 = wl.cap - steps - 3
    cache = fill_cache(dms, W, wl, n0, device, kv_format="fp8")
    qs, ks, vs, ls = step_inputs(W, wl, n0, steps + 3, device)
    out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device=device)

    def step(i):
        rc = lib.dms_step(cache.handle, ks[i].data_ptr(), vs[i].data_ptr(), ls[i].data_ptr(), qs[i].data_ptr(),
                          out.data_ptr(), wl.scale, wl.Hq, stream.cuda_stream)
        if rc:
            raise dms.DmsError(rc, "dms_step (fp8)")

    for i in range(3):
        step(i)
    torch.cuda.synchronize(device)
    len0 = int(cache.lengths().sum())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gate()
    e0.record(stream)
    for i in range(3, steps + 3):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(device)
    step_us = e0.elapsed_time(e1) * 1e3 / steps
    len1 = int(cache.lengths().sum())
    gate()
    e0.record(stream)
    for _ in range(steps):
        rc = lib.dms_decode_attention(cache.handle, qs[-1].data_ptr(), out.data_ptr(), wl.scale, wl.Hq,
                                      stream.cuda_stream)
        if rc:
            raise dms.DmsError(rc, "dms_decode_attention (fp8)")
    e1.record(stream)
    torch.cuda.synchronize(device)
    dec_us = e0.elapsed_time(e1) * 1e3 / steps
    st = cache.status()
    cache.close()
    if st != dms.DMS_OK:
        raise dms.DmsError(st, "fp8 leg")
    alg = decode_bytes_fp8(wl, len1)
    return {"storage": "fp8 e4m3, float32 scale per K row and V row", "ms_per_step": step_us * 1e-3,
            "tokens_per_s": wl.B / (step_us * 1e-6),
            "decode_us_per_launch_back_to_back": dec_us, "algorithmic_bytes_per_launch": alg,
            "achieved_GBps": alg / (dec_us * 1e-6) / 1e9,
            "kv_token_reads_per_step": 0.5 * (len0 + len1),
            "note": "step = one fused launch (the token is quantized and appended, then attended over)"}


def time_graph_leg(dms, W, device, steps):
    """The long-context stack's decode step over all its layers (one cache per
    layer, each filled to the stack's prefill length): `steps` steps as one
    dms_step call per layer, then as one launch of a DmsStepGraph holding the
    same per-layer steps.  Device time from events around each pass, host time
    of the enqueue loops from the wall clock."""
    import time as _time
    wl = W.WORKLOADS["long-context"]
    lib = dms.load_library()
    stream = torch.cuda.current_stream(device)
    caches = [fill_cache(dms, W, wl, wl.prefill, device, layer=layer) for layer in range(wl.layers)]
    ins = [step_inputs(W, wl, wl.prefill, 1, device, layer=layer) for layer in range(wl.layers)]
    qs, ks, vs, ls = ([x[j][0] for x in ins] for j in range(4))
    outs = [torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device=device) for _ in caches]

    def per_layer_step():
        for c, k, v, lg, q, o in zip(caches, ks, vs, ls, qs, outs):
            rc = lib.dms_step(c.handle, k.data_ptr(), v.data_ptr(), lg.data_ptr(), q.data_ptr(), o.data_ptr(),
                              wl.scale, wl.Hq, stream.cuda_stream)
            if rc:
                raise dms.DmsError(rc, "dms_step")

    graph = dms.DmsStepGraph(caches, ks, vs, ls, qs, outs, wl.scale)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gate()
        h0 = _time.perf_counter()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        h1 = _time.perf_counter()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / steps, (h1 - h0) * 1e6 / steps

    dev_loop, host_loop = timed(per_layer_step)
    dev_graph, host_graph = timed(lambda: graph.launch(stream))
    graph.close()
    st = [c.status() for c in caches]
    for c in caches:
        c.close()
    if any(st):
        raise dms.DmsError(max(st, key=abs), "graph leg")
    return {"workload": f"long-context stack: {wl.layers} layers, batch {wl.B}, {wl.Hq} query / {wl.Hkv} KV heads, "
                        f"head_dim {wl.D}, context {wl.prefill}", "layers": wl.layers, "steps": steps,
            "per_layer_calls": {"us_per_step_device": dev_loop, "us_per_step_host_enqueue": host_loop},
            "graph": {"us_per_step_device": dev_graph, "us_per_step_host_enqueue": host_graph},
            "tokens_per_s_graph": wl.B / (dev_graph * 1e-6)}


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1800.0, "fallback"


def prefill_flops(wl, lens, t_ctx, C):
    """Algorithmic flops of one chunk's attention: every (query row, key) pair
    the rows may attend to -- the retained cache plus the chunk's causal prefix
    -- costs 2 D for Q K^T and 2 D for P V."""
    pairs = 0
    for L in lens:  # per (sequence, KV head)
        pairs += wl.G * (C * int(L) + C * (C + 1) // 2)
    return 4 * wl.D * pairs


def time_prefill_leg(dms, W, steps, device):
    """The chunked prefill (a row of the hot path that the decode metric does not
    cover): one layer of the long-context workload, chunks of 512 tokens at a
    context of ~29-33K.  Times dms_prefill (attention + append) per chunk with
    events, and dms_append_chunk alone on a twin cache at the same positions;
    the difference is the attention kernel."""
    wl = W.WORKLOADS["long-context"]
    C = wl.chunk
    n_end = wl.prefill
    n0 = n_end - C * steps
    lib = dms.load_library()
    a = fill_cache(dms, W, wl, n0, device, layer=0)
    b = fill_cache(dms, W, wl, n0, device, layer=0)
    k, v, lg = W.kv_range(wl, 0, n0, n_end, device=device)
    q = W.q_range(wl, 0, n0, n_end, device=device)
    chunks = [(q[:, :, j * C:(j + 1) * C].contiguous(), k[:, :, j * C:(j + 1) * C].contiguous(),
               v[:, :, j * C:(j + 1) * C].contiguous(), lg[:, :, j * C:(j + 1) * C].contiguous()) for j in range(steps)]
    out = torch.empty((wl.B, wl.Hq, C, wl.D), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    t_pre, t_app, flops = [], [], 0
    for j, (qq, kk, vv, ll) in enumerate(chunks):
        lens = a.lengths().cpu().numpy().ravel()
        flops_j = prefill_flops(wl, lens, n0 + j * C, C)
        e0, e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        e0.record(stream)
        rc = lib.dms_prefill(a.handle, qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), ll.data_ptr(), C,
                             out.data_ptr(), wl.scale, wl.Hq, sh)
        e1.record(stream)
        if rc:
            raise dms.DmsError(rc, "dms_prefill")
        e2.record(stream)
        rc = lib.dms_append_chunk(b.handle, kk.data_ptr(), vv.data_ptr(), ll.data_ptr(), C, sh)
        e3.record(stream)
        if rc:
            raise dms.DmsError(rc, "dms_append_chunk")
        torch.cuda.synchronize(device)
        if j >= 1:  # the first chunk is warm-up
            t_pre.append(e0.elapsed_time(e1) * 1e3)
            t_app.append(e2.elapsed_time(e3) * 1e3)
            flops += flops_j
    st = a.status()
    if st != dms.DMS_OK:
        raise dms.DmsError(st, "device status after the prefill leg")
    a.close()
    b.close()
    n = len(t_pre)
    pre_us, app_us = sum(t_pre) / n, sum(t_app) / n
    attn_us = max(pre_us - app_us, 1e-3)
    tflops = flops / n / (attn_us * 1e-6) / 1e12
    peak, kind = measured_bf16_peak()
    return {"workload": f"long-context layer: batch {wl.B}, {wl.Hq} query / {wl.Hkv} KV heads, head_dim {wl.D}, "
                        f"chunks of {C} at context {n0 + C}..{n_end}",
            "chunks_timed": n, "us_per_chunk_call": pre_us, "us_per_chunk_append": app_us,
            "us_per_chunk_attention": attn_us, "tokens_per_s": wl.B * C / (pre_us * 1e-6),
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "peak_source": f"{kind} dense bf16 (burst)",
                         "kernel": "prefill_attention_kernel (tcgen05)",
                         "algorithmic_flops_per_chunk": flops / n,
                         "flops_definition": "4 * head_dim per (query row, key) pair over the retained cache "
                                             "and the chunk's causal prefix"}}


def workload_config(wl, n_ctx):
    return {"workload": f"{wl.name} decode at context {n_ctx}: batch {wl.B}, {wl.Hq} query / {wl.Hkv} KV heads, "
                        f"head_dim {wl.D}, window {wl.w}, eviction logits {wl.logits}",
            "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D, "window": wl.w,
            "context": n_ctx, "l2": "inputs larger than L2 (retained K/V > 126 MB), no flush"}


def run_reference(args, wl):
    rows = [0, 1]
    n_ctx = wl.cap
    run = oracle_timer(wl, n_ctx, rows)
    for i in range(args.warmup):
        run(n_ctx - 1 - (i % 256))
    t0 = time.perf_counter()
    for i in range(args.steps):
        run(n_ctx - 1 - (i % 256))
    dt = time.perf_counter() - t0
    value = len(rows) * args.steps / dt
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": workload_config(wl, n_ctx),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"each step: the oracle's decode step (mask + dense softmax attention) for "
                                   f"batch rows {rows} of {wl.B} at a position in {n_ctx - 256}..{n_ctx - 1}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="qwen3-8b")
    ap.add_argument("--no-cr1", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-storage leg")
    ap.add_argument("--no-graph", action="store_true", help="skip the multi-layer CUDA-graph step leg")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload decode table")
    ap.add_argument("--no-sweep", action="store_true", help="skip the context sweep (1K..16K)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill leg and print its figures (for profiling)")
    ap.add_argument("--prefill-chunks", type=int, default=9)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from learned_kv_cache_eviction_b300 import workload as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = W.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return

    from learned_kv_cache_eviction_b300 import dms

    if args.prefill_only:
        device = torch.device("cuda", local_rank)
        torch.cuda.set_device(device)
        print(json.dumps({"impl": "native", "prefill": time_prefill_leg(dms, W, args.prefill_chunks, device)}),
              flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist = tdist
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    # weak scaling: every rank serves its own batch of independent sequences
    wl_rank = replica_workload(wl, rank)
    n_end = wl.cap
    n0 = n_end - args.warmup - 2 * args.steps  # warm-up, pass A (timed), pass B (per-call events)
    if n0 < 1:
        ap.error("warmup + 2 * steps must be below the capacity")

    clocks = ClockSampler(device.index)  # its process starts while the cache fills
    cache = fill_cache(dms, W, wl_rank, n0, device)
    ins = step_inputs(W, wl_rank, n0, args.warmup + 2 * args.steps, device)
    r = time_device_leg(dms, cache, ins, args.warmup, args.steps, wl.scale, device, clocks, dist)
    cache.close()
    del ins
    total_ms = max_over_ranks(dist, r["total_ms"], device)

    cr1 = None
    if not args.no_cr1:
        wl1 = W.WORKLOADS["qwen3-8b-cr1"] if args.workload == "qwen3-8b" else wl_rank.with_(logits=("const", -10.0))
        wl1 = replica_workload(wl1, rank)
        c1 = fill_cache(dms, W, wl1, n0, device)
        ins1 = step_inputs(W, wl1, n0, args.warmup + 2 * args.steps, device)
        cr1 = time_device_leg(dms, c1, ins1, args.warmup, args.steps, wl.scale, device, None, dist)
        c1.close()
        del ins1

    e2e = None
    if not args.no_e2e:
        ms, h2d, d2h = time_e2e_leg(dms, W, wl_rank, n0, args.warmup, args.steps, device, dist)
        e2e = (max_over_ranks(dist, ms, device), h2d, d2h)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    len_avg = 0.5 * (r["len_sum_start"] + r["len_sum_end"])
    # the fused kernel of pass A: decode over the lengths after each step's
    # append (their mean over the pass) plus the append itself
    step_us = total_ms * 1e3 / args.steps
    alg = decode_bytes(wl, len_avg) + append_bytes(wl)
    achieved = alg / (step_us * 1e-6) / 1e9
    dec_bytes_c = decode_bytes(wl, r["len_sum_c"])
    peak, peak_kind = measured_hbm_peak()
    value = job_tokens_per_s(wl.B, args.steps, world, total_ms)
    ctx_avg = n_end - 1.5 * args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage": "bf16 K/V/q, fp32 logits/out",
        "data": "synthetic", "impl": "native",
        "config": workload_config(wl, n_end),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} HBM copy bandwidth", "traffic": profiled_traffic(),
                     "kernel": "decode_kernel<128, 4, fused> (append + decode, one launch per dms_step)",
                     "algorithmic_bytes_per_launch": alg, "us_per_launch": step_us,
                     "us_source": "mean of the timed dms_step calls (events around the pass)",
                     "frac_of_nominal_8TBps": achieved / NOMINAL_HBM_GBS},
        "decode_attention": {"us_per_launch_back_to_back": r["decode_us"],
                             "achieved_GBps": dec_bytes_c / (r["decode_us"] * 1e-6) / 1e9,
                             "frac": dec_bytes_c / (r["decode_us"] * 1e-6) / 1e9 / peak,
                             "us_per_call_events_mean": r["decode_us_call"],
                             "us_per_call_events_median": r["decode_us_call_median"],
                             "append_us_per_call_events": r["append_us_call"],
                             "note": "per-call events sit between launches and add a launch gap to each call",
                             "tokens_per_s": wl.B / (r["decode_us"] * 1e-6),
                             "kv_token_reads_per_step": len_avg,
                             "peak_tokens_in_memory": max(r["len_sum_start"], r["len_sum_end"], r["len_sum_c"]),
                             "peak_tokens_note": "the pages' second cost measure: the most KV tokens held "
                                                 "(sum of retained lengths over all sequences and KV heads) at "
                                                 "any point of the run; the retained total only grows here, so "
                                                 "it is the total after the last step",
                             "realised_cr": wl.B * wl.Hkv * ctx_avg / len_avg},
        "gpu_launches": args.steps,
        "gpu_launches_note": "per timed step: one decode_kernel launch (fused append + decode)",
        "clocks": clocks.summary(),
    }
    if cr1 is not None:
        line["cr1"] = {"decode_us_per_launch": cr1["decode_us"], "decode_us_per_call_events": cr1["decode_us_call"],
                       "ms_per_step": cr1["total_ms"] / args.steps,
                       "tokens_per_s": wl.B * args.steps / (cr1["total_ms"] * 1e-3),
                       "achieved_GBps": decode_bytes(wl, cr1["len_sum_c"]) / (cr1["decode_us"] * 1e-6) / 1e9,
                       "kv_token_reads_per_step": cr1["len_sum_c"],
                       "decode_speedup_cr8_over_cr1": cr1["decode_us"] / r["decode_us"],
                       "step_speedup_cr8_over_cr1": cr1["total_ms"] / r["total_ms"],
                       "realised_cr": cr1["len_sum_c"] / r["len_sum_c"]}
    if e2e is not None:
        ms, h2d, d2h = e2e
        line["e2e"] = {"value": job_tokens_per_s(wl.B, args.steps, world, ms), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "note": "Python API (DmsCache.step_host = dms_step_host): each step's inputs in pinned "
                               "host memory copied in on the library's copy stream, append + decode in one launch "
                               "on the compute stream, its output copied out to its own pinned buffer on a "
                               "second copy stream (every pinned buffer copied once before timing); copies of one step overlap the "
                               "neighbouring steps; timed until the last output is in host memory"}
    if not args.no_variants and world == 1:
        line["variants"] = time_variants(dms, W, device, 32)
    if not args.no_sweep and world == 1:
        line["context_sweep"] = time_context_sweep(dms, W, device)
    if not args.no_workloads and world == 1:
        line["workloads"] = time_workloads(dms, W, device, 64)
        line["literal"] = time_workloads(dms, W, device, 64, names=LITERAL_ROWS)
    if not args.no_graph and world == 1:
        line["step_graph"] = time_graph_leg(dms, W, device, 32)
    if not args.no_fp8 and world == 1:
        fp8 = time_fp8_leg(dms, W, wl, device, 64)
        fp8["decode_speedup_over_bf16"] = r["decode_us"] / fp8["decode_us_per_launch_back_to_back"]
        line["fp8"] = fp8
    if not args.no_prefill and world == 1:
        line["prefill"] = time_prefill_leg(dms, W, args.prefill_chunks, device)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, n_end)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
