"""Benchmark of the paged-attention hot path on GB300.

The headline step is the cache write of the batch's 38 new tokens fused into
paged decode (pa_decode_append: split partitions + log-sum-exp combine; the
two-launch path pa_kv_cache_write + pa_decode is timed beside it) over the
LLaMA-13B-shaped batch: 38 sequences, 40 heads, head_dim 128, block_size 16,
context lengths uniform in [128, 2048], fp16 N(0,1) synthetic data.  The
metric is algorithmic HBM GB/s (K+V rows attended + q + out + table/length
reads + the cache write's read and write), plus attended tokens/s.

The same JSON line carries a ``workloads`` object with the other paged-
attention workloads, each timed the same way (CUDA events on the launching
stream, L2 flushed before every timed step) with its roofline fraction,
DRAM traffic (when a capture of the current source exists), clock record and
the fp64 oracle timed on one pinned host core on a bounded sample:
  prefix_sharing      -- 16 prompts x 8 samples, block copy + grouped decode
  long_context        -- one 1,048,576-token sequence, split-KV decode
  chunked_prefill     -- 8 x 512-query chunks on 3,584 cached tokens (tcgen05)
  llama13b_decode_fp8 -- the 38-sequence batch stored as e4m3

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME]  (one workload on its own line)

Multi-GPU (torchrun): every rank runs its own independent batch (decode
sequences are independent; no collective on the data path); value = bytes
of all ranks / max-over-ranks time, scaling "weak".
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (rank 0 only).
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from contextlib import contextmanager

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged-decode KV HBM GB/s (% of ~8 TB/s) and attended tokens/s, 1×GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of a workload's
# dominant kernel, from one ncu capture (profiles/), keyed by the workload, the
# block size and the hash of the sources that kernel is built from; null once
# any of them changes.
TRAFFIC = {
    # partition_kernel<128,16,4,2,fp16> with the fused write, 38-sequence step
    ("llama13b_decode", 16, "6926943ee2a6ce18"): 853313280 + 5961984,
    # the grouped partition kernel of the 16 x 8 prefix-sharing batch
    ("prefix_sharing", 16, "6926943ee2a6ce18"): 1093610240 + 10890240,
    # partition kernel over a 65,536-token context, scaled by tokens (x16)
    ("long_context", 16, "6926943ee2a6ce18"): (1342285568 + 6882304) * 16,
    # the e4m3 partition kernel (two heads per warp), 38-sequence batch
    ("llama13b_decode_fp8", 16, "6926943ee2a6ce18"): 439972608 + 4957440,
    # prefill_kernel<128,16>, 8 x 512 queries on 3,584 cached tokens
    ("chunked_prefill", 16, "974571cd2e30d09f"): 713150976 + 36221184,
}
TRAFFIC_SOURCES = {
    "llama13b_decode": ("decode.cu", "pk_common.cuh", "pk_prefix.cuh", "pk_internal.h"),
    "prefix_sharing": ("decode.cu", "pk_common.cuh", "pk_prefix.cuh", "pk_internal.h"),
    "long_context": ("decode.cu", "pk_common.cuh", "pk_prefix.cuh", "pk_internal.h"),
    "llama13b_decode_fp8": ("decode.cu", "pk_common.cuh", "pk_prefix.cuh", "pk_internal.h"),
    "chunked_prefill": ("prefill.cu", "pk_common.cuh", "pk_tcgen05.cuh", "pk_internal.h"),
}


def src_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_172_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(workload, block_size):
    return TRAFFIC.get((workload, block_size, src_hash(TRAFFIC_SOURCES[workload])))


def measured_peaks():
    """(HBM GB/s, kind), (dense fp16/bf16 TFLOP/s burst, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), "measured"), (float(d["bf16_tflops"]), "measured")
    except Exception:
        return (FALLBACK_HBM_GBS, "fallback"), (FALLBACK_BF16_TFLOPS, "fallback")


# ---------------------------------------------------------------------------
# byte and FLOP accounting
# ---------------------------------------------------------------------------
def decode_bytes(ctx, B, H, D, bs, elem_bytes=2, scale_bytes=0):
    """K+V rows attended (+ per-row scales) + q + out + table/length reads."""
    ctx = np.asarray(ctx, dtype=np.int64)
    kv = int(ctx.sum()) * H * (2 * D * elem_bytes + 2 * scale_bytes)
    qo = 2 * B * H * D * 2
    tables = int(sum(-(-int(c) // bs) for c in ctx)) * 4 + B * 4
    return kv + qo + tables


def write_bytes(T, H, D):
    return 2 * (2 * T * H * D * 2) + T * 8


def prefill_flops(ctx, Lq, H, D):
    """Useful causal FLOPs: query i of the chunk sees ctx-Lq+i+1 keys; each
    (query, key) pair costs 2*D for Q K^T and 2*D for P V."""
    total = 0
    for n in ctx:
        n = int(n)
        total += Lq * (n - Lq + 1) + Lq * (Lq - 1) // 2
    return 4 * D * H * total


def unique_kv_bytes(tables, ctx, bs, H, D):
    """K+V bytes of the distinct physical rows the batch attends to."""
    used = {}
    for b, n in enumerate(ctx):
        n = int(n)
        for lb in range(-(-n // bs)):
            phys = int(tables[b, lb])
            used[phys] = max(used.get(phys, 0), min(bs, n - lb * bs))
    return sum(used.values()) * H * D * 2 * 2


# ---------------------------------------------------------------------------
# clocks during the timed regions (read-only NVML queries; nvidia-smi fallback)
# ---------------------------------------------------------------------------
_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


class Nvml:
    """Read-only NVML queries through ctypes (no settings are changed)."""

    def __init__(self, device):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.handle = ctypes.c_void_p()
        rc = -1
        try:
            bus = torch.cuda.get_device_properties(device).pci_bus_id
            dom = torch.cuda.get_device_properties(device).pci_domain_id
            dv = torch.cuda.get_device_properties(device).pci_device_id
            pci = f"{dom:08x}:{bus:02x}:{dv:02x}.0".encode()
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci, ctypes.byref(self.handle))
        except Exception:
            rc = -1
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(
                ctypes.c_uint(torch.device(device).index or 0), ctypes.byref(self.handle))
        if rc != 0:
            raise RuntimeError(f"no NVML handle ({rc})")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        sm, mx = ctypes.c_uint(), ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(sm)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))
        self._reasons(self.handle, ctypes.byref(r))
        return float(sm.value), float(mx.value), int(r.value)


class ClockSampler:
    """Polls the SM clock and the clock-event reasons every ~5 ms (NVML) from
    a thread; summary() reports the samples that fall inside given windows
    (the timed regions, as perf_counter intervals)."""

    def __init__(self, device):
        self.samples = []  # (perf_counter time, sm MHz, max MHz, reasons mask)
        self.note = None
        self._stop = threading.Event()
        self._proc = None
        try:
            self.nvml = Nvml(device)
        except Exception as e:  # fall back to the nvidia-smi loop
            self.nvml = None
            self.note = f"NVML unavailable ({e!r}); nvidia-smi -lms 20"
        self.device = device

    def start(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
        else:
            idx = torch.device(self.device).index or 0
            fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,"
                      "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(idx), f"--query-gpu={fields}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            except Exception as e:
                self.note = (self.note or "") + f"; nvidia-smi failed to start ({e!r})"
                self._proc = None
            self._thread = threading.Thread(target=self._read_smi, daemon=True)
        self._thread.start()
        return self

    def _poll(self):
        while not self._stop.is_set():
            s = self.nvml.sample()
            if s is not None:
                self.samples.append((time.perf_counter(),) + s)
            time.sleep(0.005)

    def _read_smi(self):
        if self._proc is None:
            return
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            mask = 0
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    mask |= _REASON_BITS[n]
            self.samples.append((time.perf_counter(), sm, mx, mask))

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                _, err = self._proc.communicate(timeout=5)
                if not self.samples:
                    self.note = (self.note or "") + \
                        f"; nvidia-smi rc={self._proc.returncode} stderr={err.strip()[:200]!r}"
            except Exception:
                self._proc.kill()
        self._thread.join(timeout=2)

    def summary(self, windows):
        """Median SM clock, max clock and active reasons over the samples taken
        inside the given (t0, t1) perf_counter windows."""
        sel = [s for s in self.samples if any(t0 <= s[0] <= t1 for t0, t1 in windows)]
        out = {"samples": len(sel), "source": "nvml" if self.nvml is not None else "nvidia-smi"}
        if self.note:
            out["note"] = self.note
        if not sel:
            out.update({"sm_mhz": None, "sm_max_mhz": None, "reasons": []})
            return out
        mask = 0
        for s in sel:
            mask |= s[3]
        out.update({"sm_mhz": statistics.median(s[1] for s in sel),
                    "sm_min_mhz": min(s[1] for s in sel),
                    "sm_max_mhz": max(s[2] for s in sel),
                    "reasons": sorted(n for n, b in _REASON_BITS.items() if mask & b)})
        return out


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------
class Flusher:
    """Evicts the previous step from L2 between timed steps (untimed): reads a
    buffer 4x the L2 size, so L2 ends up holding clean lines only and no
    write-back of flush data lands in the timed region."""

    def __init__(self, dev):
        self.buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        torch.sum(self.buf, dim=0, out=self.sink)


def timed_steps(phases, stream, flush, K, warmup, sustain_s=0.0, barrier=None):
    """Warm-up, then K steps, each bracketed (per phase) by CUDA events on
    `stream` with an L2 flush before it; the K steps are bracketed by
    `barrier` (if given) and a device synchronisation on both sides.  Returns
    per-phase mean ms, per-step ms, the perf_counter windows of the timed
    regions, and (sustain_s > 0) the mean ms of the same steps run back to
    back for sustain_s seconds of wall time (the clock window)."""
    def run(evs=None):
        for i, (_, fn) in enumerate(phases):
            if evs is not None:
                evs[i].record(stream)
            fn()
        if evs is not None:
            evs[-1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            run()
    torch.cuda.synchronize()
    n = len(phases)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(K)]
    if barrier is not None:
        barrier()
        torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush()
            run(evs[i])
    torch.cuda.synchronize()
    windows = [(t0, time.perf_counter())]
    if barrier is not None:
        barrier()
    phase_ms = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, (nm, _) in enumerate(phases)}
    step_ms = [e[0].elapsed_time(e[-1]) for e in evs]
    sustained = None
    if sustain_s > 0:
        sev = []
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - t0 < sustain_s:
                for _ in range(16):
                    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                    flush()
                    e[0].record(stream)
                    run()
                    e[1].record(stream)
                    sev.append(e)
                if len(sev) >= 64:  # keep the host no more than a few steps ahead
                    sev[-64][1].synchronize()
        torch.cuda.synchronize()
        windows.append((t0, time.perf_counter()))
        sustained = {"ms_per_step": statistics.mean(a.elapsed_time(b) for a, b in sev),
                     "steps": len(sev)}
    return phase_ms, step_ms, windows, sustained


# ---------------------------------------------------------------------------
# the oracle on one pinned host core
# ---------------------------------------------------------------------------
@contextmanager
def one_core():
    """Pins this thread to one core of its current affinity set for the
    duration; yields what the CPU baseline reports about the host."""
    info = {"cpu_count": os.cpu_count()}
    prev = None
    try:
        prev = sorted(os.sched_getaffinity(0))
        info["affinity"] = prev
        core = prev[-1]
        os.sched_setaffinity(0, {core})
        info["pinned_core"] = core
    except (AttributeError, OSError):
        info["affinity"] = None
        info["pinned_core"] = None
    try:
        yield info
    finally:
        if prev is not None:
            try:
                os.sched_setaffinity(0, set(prev))
            except OSError:
                pass


def cpu_line(value, unit, seconds, sample, info, scaled):
    d = {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "seconds": seconds,
         "sample": sample, "cpu_count": info["cpu_count"], "affinity": info["affinity"],
         "pinned_core": info["pinned_core"]}
    if scaled:
        d["scaling"] = scaled
    return d


def compact_pool(tables, ctx, bs, pools, extra_blocks=()):
    """The physical blocks the first len(ctx) sequences attend to (plus
    extra_blocks), gathered on the device into a pool holding only them,
    returned as host numpy arrays; tables renumbered (-1 past each sequence)
    and the old -> new block map."""
    used = set(int(x) for x in extra_blocks)
    for b in range(len(ctx)):
        used.update(int(x) for x in tables[b, :-(-int(ctx[b]) // bs)])
    uniq = sorted(used)
    remap = {old: new for new, old in enumerate(uniq)}
    out = []
    for p in pools:
        idx = torch.as_tensor(uniq, dtype=torch.int64, device=p.device)
        out.append(p.index_select(0, idx).cpu().contiguous().numpy())
    bt2 = np.full((len(ctx), tables.shape[1]), -1, dtype=np.int32)
    for b in range(len(ctx)):
        nb = -(-int(ctx[b]) // bs)
        bt2[b, :nb] = [remap[int(x)] for x in tables[b, :nb]]
    return out, bt2, remap


def sequences_within(per_key_s, ctx, budget_s):
    n = 1
    while n < len(ctx) and per_key_s * float(np.sum(ctx[:n + 1])) < budget_s:
        n += 1
    return n


# ---------------------------------------------------------------------------
# the headline step: 38-sequence decode with the fused cache write
# ---------------------------------------------------------------------------
def make_workload(device, seed=1, block_size=16):
    from paged_kv_cache_172_gb300 import workloads
    return workloads.llama13b_decode(seed=seed, device=device, block_size=block_size)


def workload_config(batch):
    """The workload, identical in both arms (no launch or timing keys)."""
    ctx = batch.context_lens.cpu().numpy()
    return {"workload": f"llama13b_decode_b38: 38 seqs x 40 heads x head_dim 128, block_size "
                        f"{batch.block_size}, context_lens U[128,2048] (seed 1), pool 1.2x "
                        "need, randomly permuted blocks; step = cache write of 38 new tokens "
                        "fused into decode (pa_decode_append)",
            "B": int(batch.B), "H": int(batch.H), "head_dim": int(batch.D),
            "block_size": int(batch.block_size), "num_blocks": int(batch.num_blocks),
            "sum_context_len": int(ctx.sum())}


def run_gpu(args, rank, world, local_rank):
    import paged_kv_cache_172_gb300 as pk
    from paged_kv_cache_172_gb300.session import DecodeSession

    dev = torch.device("cuda", local_rank)
    batch = make_workload(dev, seed=1 + rank, block_size=args.block_size)
    B, H, D, bs = batch.B, batch.H, batch.D, batch.block_size
    ctx = batch.context_lens.cpu().numpy()
    max_ctx = 2048
    pt = args.partition_tokens or pk.pa_decode_partition_tokens(B, H, bs, max_ctx)
    ws_bytes = pk.pa_decode_workspace_size(B, H, D, bs, max_ctx, pt)
    ws = torch.empty(max(ws_bytes // 4, 1) + 4, dtype=torch.float32, device=dev)
    out = torch.empty_like(batch.q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    flush = Flusher(dev)

    def step():
        # the 38 new tokens' cache write fused into the decode launch
        pk.pa_decode_append(batch.q, batch.k_new, batch.v_new, batch.k_cache, batch.v_cache,
                            batch.block_tables, batch.context_lens, batch.scale, max_ctx,
                            out=out, partition_tokens=pt, workspace=ws, status=status,
                            stream=stream)

    def write_unfused():
        pk.pa_kv_cache_write(batch.k_new, batch.v_new, batch.slot_mapping, batch.k_cache,
                             batch.v_cache, status=status, stream=stream)

    def decode_unfused():
        pk.pa_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                     batch.context_lens, batch.scale, max_ctx, out=out, partition_tokens=pt,
                     workspace=ws, status=status, stream=stream)

    n_parts = -(-max_ctx // pt)
    launches_per_step = 1 + (1 if n_parts > 1 else 0)
    K = args.steps
    _, step_ms, windows, _ = timed_steps([("step", step)], stream, flush, K, args.warmup,
                                         barrier=torch.distributed.barrier if world > 1 else None)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the timed region")
    total_ms = sum(step_ms)
    # the clock window: the same step back to back (sampled, not the headline)
    _, _, cwin, sustained = timed_steps([("step", step)], stream, flush, 1, 1,
                                        sustain_s=args.clock_window_s)
    windows += cwin[1:]

    # -- the same step as two launches (cache write, then decode), for reference
    pm, unfused_ms, w2, _ = timed_steps([("write", write_unfused), ("decode", decode_unfused)],
                                        stream, flush, K, args.warmup)
    windows += w2

    # -- end to end: host buffers, copies inside the timed region ---------------
    # Zero copy (the session's default): the kernels load every input from
    # pinned host memory and store out there.  Staged: one copy in, one out.
    step()
    torch.cuda.synchronize(dev)
    ref_out = out.cpu()
    e2e = {}
    for zero_copy in (True, False):
        sess = DecodeSession(batch.k_cache, batch.v_cache, B, batch.block_tables.shape[1],
                             max_ctx, batch.scale, partition_tokens=pt, zero_copy=zero_copy)
        host = sess.host_buffers()
        host["q"].copy_(batch.q)
        host["k_new"].copy_(batch.k_new)
        host["v_new"].copy_(batch.v_new)
        host["context_lens"].copy_(batch.context_lens)
        host["block_tables"].copy_(batch.block_tables)
        _, ms, w3, _ = timed_steps([("e2e", lambda: sess.step_from_host(
            host, status=status, stream=stream))], stream, flush, K, args.warmup)
        windows += w3
        if not torch.equal(host["out"], ref_out):
            raise RuntimeError("end-to-end output differs from the device-resident run")
        # host wall clock of the same call: the ctypes marshalling and launches,
        # the transfers and kernels, and the stream synchronisation before the
        # caller can read host['out'] (the L2 flush before each step untimed)
        wall = []
        for _ in range(K):
            with torch.cuda.stream(stream):
                flush()
            stream.synchronize()
            t0 = time.perf_counter()
            sess.step_from_host(host, status=status, stream=stream)
            stream.synchronize()
            wall.append((time.perf_counter() - t0) * 1e3)
        e2e[zero_copy] = (sum(ms) / K, sess.h2d_bytes(), sess.d2h_bytes(),
                          statistics.mean(wall), statistics.median(wall))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x}")

    dbytes = decode_bytes(ctx, B, H, D, bs)
    sbytes = dbytes + write_bytes(int(batch.slot_mapping.numel()), H, D)
    return {
        "step_ms": total_ms / K, "step_ms_median": statistics.median(step_ms),
        "sustained": sustained,
        "decode_ms": pm["decode"], "write_ms": pm["write"],
        "unfused_ms": statistics.mean(unfused_ms),
        "e2e": e2e, "step_bytes": sbytes, "decode_bytes": dbytes,
        "tokens": int(ctx.sum()), "windows": windows, "partition_tokens": pt,
        "num_parts": n_parts, "launches": launches_per_step * K, "batch": batch,
    }


def cpu_baseline(batch, budget_s):
    """The fp64 oracle on one pinned core on a bounded sample of the headline
    step: the cache write of the new tokens, then decode of the first
    sequences whose estimated cost fits ``budget_s``."""
    import oracle
    H, D, bs = batch.H, batch.D, batch.block_size
    ctx = batch.context_lens.cpu().numpy()
    bt = batch.block_tables.cpu().numpy()
    sm = batch.slot_mapping.cpu().numpy()
    kn, vn = batch.k_new.cpu().numpy(), batch.v_new.cpu().numpy()
    q = batch.q.cpu().numpy()
    with one_core() as info:
        (kc1, vc1), bt1, _ = compact_pool(bt, ctx[:1], bs, [batch.k_cache, batch.v_cache])
        t0 = time.perf_counter()
        oracle.decode(q[:1], kc1, vc1, bt1, ctx[:1], batch.scale)
        per_key = (time.perf_counter() - t0) / max(int(ctx[0]), 1)
        n = sequences_within(per_key, ctx, budget_s)
        kc = batch.k_cache.cpu().numpy()
        vc = batch.v_cache.cpu().numpy()
        t0 = time.perf_counter()
        kc2, vc2 = oracle.kv_cache_write(kn, vn, sm, kc, vc)
        oracle.decode(q[:n], kc2, vc2, bt[:n], ctx[:n], batch.scale)
        dt = time.perf_counter() - t0
    byts = decode_bytes(ctx[:n], n, H, D, bs) + write_bytes(len(sm), H, D)
    return cpu_line(byts / dt / 1e9, "GB/s", dt,
                    f"cache write of {len(sm)} tokens + decode of the first {n} of {len(ctx)} "
                    f"sequences ({int(ctx[:n].sum())} keys x {H} heads), fp64, one thread "
                    "pinned to one core", info, None)


# ---------------------------------------------------------------------------
# the other workloads: specs, timing, their CPU samples
# ---------------------------------------------------------------------------
WORKLOADS = ("prefix_sharing", "long_context", "chunked_prefill", "llama13b_decode_fp8")


def spec_prefix_sharing(pk, workloads, dev, args, status, stream):
    batch = workloads.prefix_sharing(seed=2, device=dev)
    lay = batch.meta["layout"]
    ctx = lay.context_lens
    max_ctx = int(ctx.max())
    out = torch.empty_like(batch.q)
    H, D, bs = batch.H, batch.D, batch.block_size
    sg, off, seqs, pref = (torch.from_numpy(x).to(dev) for x in workloads.sharing_groups(lay))
    max_prefix = int(pref.max())
    pt = max_prefix // 3  # 336: three partitions cover the 1,008 shared tokens
    phases = [
        ("block_copy", lambda: pk.pa_block_copy(batch.k_cache, batch.v_cache, batch.copy_pairs,
                                                status=status, stream=stream)),
        ("decode", lambda: pk.pa_decode_shared_prefix(
            batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.context_lens, sg,
            off, seqs, pref, batch.scale, max_ctx, 8, max_prefix, out=out, partition_tokens=pt,
            status=status, stream=stream)),
    ]
    alt = {"decode_without_sharing": lambda: pk.pa_decode(
        batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.context_lens,
        batch.scale, max_ctx, out=out, status=status, stream=stream)}
    logical = decode_bytes(ctx, batch.B, H, D, bs)
    unique = unique_kv_bytes(lay.tables, ctx, bs, H, D) + 2 * batch.B * H * D * 2
    copy_bytes = 2 * 2 * len(lay.pairs) * bs * H * D * 2

    def cpu_sample(budget_s):
        import oracle
        pairs = lay.pairs
        q = batch.q.cpu().numpy()
        with one_core() as info:
            def run(n):
                (kc, vc), bt2, remap = compact_pool(lay.tables, ctx[:n], bs,
                                                    [batch.k_cache, batch.v_cache],
                                                    extra_blocks=pairs[:n].ravel())
                p2 = np.array([[remap[int(s)], remap[int(d)]] for s, d in pairs[:n]], np.int64)
                t0 = time.perf_counter()
                kc, vc = oracle.block_copy(kc, vc, p2)
                oracle.decode(q[:n], kc, vc, bt2, ctx[:n], batch.scale)
                return time.perf_counter() - t0
            per_key = run(1) / float(ctx[0])
            n = sequences_within(per_key, ctx, budget_s)
            dt = run(n)
        full_s = dt * float(ctx.sum()) / float(ctx[:n].sum())
        return cpu_line(unique / full_s / 1e9, "GB/s", dt,
                        f"block copy of {n} copy-on-write pairs + decode of the first {n} of "
                        f"{len(ctx)} sequences ({int(ctx[:n].sum())} keys x {H} heads), fp64, "
                        "one thread pinned to one core", info,
                        "seconds scaled to the whole step by attended keys "
                        f"(x{float(ctx.sum()) / float(ctx[:n].sum()):.2f}); value = the step's "
                        "unique bytes over that time")

    return {
        "phases": phases, "alt": alt, "main": "decode", "work": unique, "unit": "GB/s",
        "bound": "hbm", "tokens": int(ctx.sum()), "cpu_sample": cpu_sample,
        "extra": {"logical_bytes": logical, "unique_bytes": unique, "copy_bytes": copy_bytes},
        "desc": ("prefix_sharing_16x8: 16 prompts x 8 samples, 1024-token shared prompts, "
                 "tails U[1,512], 40 heads, head_dim 128, block_size 16; step = block_copy of "
                 "128 copy-on-write blocks + pa_decode_shared_prefix (groups of 8 sharing 1,008 "
                 "tokens, 336-token partitions); GB/s on unique bytes"),
        "kernel": "pa_decode_shared_prefix (grouped partition kernel + combine)",
        "launches": 1 + 2, "block_size": bs, "batch": batch,
    }


def spec_long_context(pk, workloads, dev, args, status, stream):
    batch = workloads.long_context(seed=3, device=dev, bs=args.block_size,
                                   context_len=args.context_len)
    n = int(batch.context_lens[0])
    out = torch.empty_like(batch.q)
    H, D, bs = batch.H, batch.D, batch.block_size
    pt = pk.pa_decode_partition_tokens(1, H, bs, n)
    phases = [("decode", lambda: pk.pa_decode(batch.q, batch.k_cache, batch.v_cache,
                                              batch.block_tables, batch.context_lens,
                                              batch.scale, n, out=out, status=status,
                                              stream=stream))]
    work = decode_bytes([n], 1, H, D, bs)

    def cpu_sample(budget_s):
        import oracle
        bt = batch.block_tables.cpu().numpy()
        heads = []
        dt = 0.0
        with one_core() as info:
            for h in range(H):
                kc = batch.k_cache[:, :, h:h + 1].contiguous().cpu().numpy()
                vc = batch.v_cache[:, :, h:h + 1].contiguous().cpu().numpy()
                q = batch.q[:, h:h + 1].contiguous().cpu().numpy()
                t0 = time.perf_counter()
                oracle.decode(q, kc, vc, bt, np.array([n], np.int32), batch.scale)
                dt += time.perf_counter() - t0
                heads.append(h)
                if dt * (len(heads) + 1) / len(heads) > budget_s:
                    break
        full_s = dt * H / len(heads)
        return cpu_line(work / full_s / 1e9, "GB/s", dt,
                        f"decode of head(s) {heads} of {H} over all {n} keys, fp64, one thread "
                        "pinned to one core", info,
                        f"seconds scaled to all heads (x{H / len(heads):.1f})")

    return {
        "phases": phases, "alt": {}, "main": "decode", "work": work, "unit": "GB/s",
        "bound": "hbm", "tokens": n, "cpu_sample": cpu_sample,
        "extra": {"partition_tokens": pt, "num_parts": -(-n // pt)},
        "desc": (f"long_context: 1 sequence of {n:,} tokens, 40 heads, head_dim 128, "
                 f"block_size {bs}, {batch.num_blocks} permuted blocks "
                 f"({n * H * D * 4 / 1e9:.1f} GB K+V); split-KV decode + log-sum-exp combine"),
        "kernel": "pa_decode (partition kernel + combine)", "launches": 2, "block_size": bs,
        "batch": batch,
    }


def spec_chunked_prefill(pk, workloads, dev, args, status, stream):
    batch = workloads.chunked_prefill(seed=4, device=dev, block_size=args.block_size)
    ctx = batch.context_lens.cpu().numpy()
    out = torch.empty_like(batch.q)
    B, H, Lq, D = batch.q.shape
    bs = batch.block_size
    pws = pk.pa_prefill_workspace_size(B, H, Lq, D)
    prefill_ws = torch.empty(max(pws // 4, 1) + 4, dtype=torch.float32, device=dev)
    phases = [
        ("kv_cache_write", lambda: pk.pa_kv_cache_write(batch.k_new, batch.v_new,
                                                        batch.slot_mapping, batch.k_cache,
                                                        batch.v_cache, status=status,
                                                        stream=stream)),
        ("prefill", lambda: pk.pa_prefill_chunk(batch.q, batch.k_cache, batch.v_cache,
                                                batch.block_tables, batch.context_lens,
                                                batch.scale, out=out, workspace=prefill_ws,
                                                status=status, stream=stream)),
    ]
    work = prefill_flops(ctx, Lq, H, D)

    def cpu_sample(budget_s):
        import oracle
        bt = batch.block_tables.cpu().numpy()
        rows, dt = 16, 0.0
        with one_core() as info:
            kc = batch.k_cache[:, :, :1].contiguous().cpu().numpy()
            vc = batch.v_cache[:, :, :1].contiguous().cpu().numpy()
            while True:
                q = batch.q[:1, :1, Lq - rows:].contiguous().cpu().numpy()
                t0 = time.perf_counter()
                oracle.prefill(q, kc, vc, bt[:1], ctx[:1], batch.scale)
                dt = time.perf_counter() - t0
                if dt * 2 > budget_s or rows * 2 > Lq:
                    break
                rows *= 2
        n = int(ctx[0])
        flops = 4 * D * sum(n - rows + i + 1 for i in range(rows))
        return cpu_line(flops / dt / 1e12, "TFLOP/s", dt,
                        f"the last {rows} of the {Lq} chunk queries of sequence 0, head 0, "
                        f"against its {n} keys ({flops / 1e9:.2f} GFLOP), fp64, one thread "
                        "pinned to one core", info,
                        "value = the sample's useful FLOPs over its time (the rate is the same "
                        "for the whole step)")

    return {
        "phases": phases, "alt": {}, "main": "prefill", "work": work, "unit": "TFLOP/s",
        "bound": "tensor", "tokens": int(B * Lq), "cpu_sample": cpu_sample,
        "extra": {"useful_flops": work, "kv_bytes": int(ctx.sum()) * H * D * 4,
                  "q_out_bytes": 2 * batch.q.numel() * 2,
                  "write_bytes": write_bytes(int(batch.slot_mapping.numel()), H, D)},
        "desc": (f"chunked_prefill_8x512_on_3584: 8 sequences, 512-query chunk on 3,584 cached "
                 f"tokens (context 4,096), 40 heads, head_dim 128, block_size {bs}; step = "
                 "kv_cache_write of the 4,096 chunk tokens + pa_prefill_chunk"),
        "kernel": "pa_prefill_chunk (tcgen05 prefill kernel + tail-split combine)",
        "launches": 3, "block_size": bs, "batch": batch,
    }


def spec_fp8(pk, workloads, dev, args, status, stream):
    batch = make_workload(dev, seed=1, block_size=args.block_size)
    NB, bs, H, D = batch.k_cache.shape
    k8 = torch.zeros((NB, bs, H, D), dtype=torch.uint8, device=dev)
    v8 = torch.zeros_like(k8)
    ks = torch.ones((NB, H, bs), dtype=torch.float32, device=dev)
    vs = torch.ones_like(ks)
    all_slots = torch.arange(NB * bs, dtype=torch.int64, device=dev)
    pk.pa_kv_cache_write_fp8(batch.k_cache.reshape(NB * bs, H, D),
                             batch.v_cache.reshape(NB * bs, H, D), all_slots, k8, v8, ks, vs,
                             status=status)  # quantize the whole pool once (untimed)
    del all_slots
    out = torch.empty_like(batch.q)
    ctx = batch.context_lens.cpu().numpy()
    T = int(batch.slot_mapping.numel())
    phases = [
        ("kv_cache_write_fp8", lambda: pk.pa_kv_cache_write_fp8(
            batch.k_new, batch.v_new, batch.slot_mapping, k8, v8, ks, vs, status=status,
            stream=stream)),
        ("decode", lambda: pk.pa_decode_fp8(batch.q, k8, v8, ks, vs, batch.block_tables,
                                            batch.context_lens, batch.scale, 2048, out=out,
                                            status=status, stream=stream)),
    ]
    # e4m3 K and V rows (D bytes each) and their two fp32 scales, + q/out/tables
    work = decode_bytes(ctx, batch.B, H, D, bs, elem_bytes=1, scale_bytes=4)

    def cpu_sample(budget_s):
        import oracle
        bt = batch.block_tables.cpu().numpy()
        sm = batch.slot_mapping.cpu().numpy()
        kn, vn = batch.k_new.cpu().numpy(), batch.v_new.cpu().numpy()
        q = batch.q.cpu().numpy()

        def run(n):
            (a8, b8, sa, sb), bt2, remap = compact_pool(bt, ctx[:n], bs, [k8, v8, ks, vs])
            sm2 = np.array([remap[int(s) // bs] * bs + int(s) % bs for s in sm[:n]], np.int64)
            t0 = time.perf_counter()
            a8, b8, sa, sb = oracle.kv_cache_write_fp8(kn[:n], vn[:n], sm2, a8, b8, sa, sb)
            oracle.decode_fp8(q[:n], a8, b8, sa, sb, bt2, ctx[:n], batch.scale)
            return time.perf_counter() - t0

        with one_core() as info:
            per_key = run(1) / float(ctx[0])
            n = sequences_within(per_key, ctx, budget_s)
            dt = run(n)
        full_s = dt * float(ctx.sum()) / float(ctx[:n].sum())
        return cpu_line(work / full_s / 1e9, "GB/s", dt,
                        f"quantizing write of {n} new tokens + fp8 decode of the first {n} of "
                        f"{len(ctx)} sequences ({int(ctx[:n].sum())} keys x {H} heads), fp64, "
                        "one thread pinned to one core", info,
                        "seconds scaled to the whole step by attended keys "
                        f"(x{float(ctx.sum()) / float(ctx[:n].sum()):.2f})")

    return {
        "phases": phases, "alt": {}, "main": "decode", "work": work, "unit": "GB/s",
        "bound": "hbm", "tokens": int(ctx.sum()), "cpu_sample": cpu_sample,
        "extra": {"fp8_algorithmic_bytes": work,
                  "fp16_equivalent_bytes": decode_bytes(ctx, batch.B, H, D, bs),
                  "write_fp8_bytes": T * H * (2 * 2 * D + 2 * D + 8)},
        "desc": ("llama13b_decode_b38_fp8: the 38-sequence batch stored as e4m3 with "
                 "per-(token, head) fp32 scales; step = quantizing write of 38 new tokens + "
                 "pa_decode_fp8; GB/s on fp8 bytes"),
        "kernel": "pa_decode_fp8 (e4m3 partition kernel + combine)", "launches": 3,
        "block_size": bs, "batch": batch,
    }


SPECS = {"prefix_sharing": spec_prefix_sharing, "long_context": spec_long_context,
         "chunked_prefill": spec_chunked_prefill, "llama13b_decode_fp8": spec_fp8}


def measure_workload(name, args, dev, sampler, peaks, cpu_budget_s):
    """One workload: setup, K timed steps, its clock window, the alternatives,
    then the oracle sample.  Returns the entry of the ``workloads`` object."""
    import paged_kv_cache_172_gb300 as pk
    from paged_kv_cache_172_gb300 import workloads

    stream = torch.cuda.Stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = Flusher(dev)
    spec = SPECS[name](pk, workloads, dev, args, status, stream)
    torch.cuda.synchronize(dev)
    phase_ms, step_ms, windows, sustained = timed_steps(
        spec["phases"], stream, flush, args.steps, args.warmup, sustain_s=args.clock_window_s)
    alt_ms = {}
    for nm, fn in spec["alt"].items():  # alternatives timed beside the step, same flushing
        pm, _, w, _ = timed_steps([(nm, fn)], stream, flush, args.steps, args.warmup)
        windows += w
        alt_ms[f"{nm}_ms"] = pm[nm]
    if int(status.item()) != 0:
        raise RuntimeError(f"{name}: device status {int(status.item()):#x}")
    main_s = phase_ms[spec["main"]] / 1e3
    (hbm, hbm_kind), (tf, tf_kind) = peaks
    if spec["bound"] == "tensor":
        achieved = spec["work"] / main_s / 1e12
        peak, peak_kind = tf, f"{tf_kind} bf16 dense burst (fp16 dense rate equal)"
    else:
        achieved = spec["work"] / main_s / 1e9
        peak, peak_kind = hbm, f"{hbm_kind} HBM copy"
    entry = {
        "workload": spec["desc"], "metric": f"{name} {spec['unit']}", "value": achieved,
        "unit": spec["unit"], "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_ms), "phase_ms": phase_ms,
        "l2": "flushed before every timed step (512 MB read, untimed)",
        "roofline": {"bound": spec["bound"], "kernel": spec["kernel"], "phase": spec["main"],
                     "achieved": achieved, "peak": peak, "unit": spec["unit"],
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic_for(name, spec["block_size"]),
                     ("algorithmic_flops" if spec["bound"] == "tensor" else "algorithmic_bytes"):
                         spec["work"]},
        "tokens_per_s": spec["tokens"] / main_s,
        "gpu_launches": spec["launches"] * args.steps,
        "sustained": sustained,
        "clocks": sampler.summary(windows) if sampler else None,
    }
    entry.update(spec["extra"])
    entry.update(alt_ms)
    if name == "prefix_sharing":
        entry["logical_GBs"] = spec["extra"]["logical_bytes"] / main_s / 1e9
        entry["block_copy_GBs"] = spec["extra"]["copy_bytes"] / (phase_ms["block_copy"] / 1e3) / 1e9
    if name == "chunked_prefill":
        entry["kv_cache_write_GBs"] = spec["extra"]["write_bytes"] / \
            (phase_ms["kv_cache_write"] / 1e3) / 1e9
    if cpu_budget_s > 0:
        entry["cpu_baseline"] = spec["cpu_sample"](cpu_budget_s)
    del spec
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return entry


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def compact_sample(batch, n, heads=None):
    """The first n sequences of the batch (and only the first `heads` heads)
    on a pool holding only their blocks, tables and slots renumbered, so a
    CPU step costs in proportion to the sample."""
    bs = batch.block_size
    hh = batch.H if heads is None else heads
    ctx = batch.context_lens.cpu().numpy()[:n]
    bt = batch.block_tables.cpu().numpy()[:n]
    (kc, vc), bt2, remap = compact_pool(bt, ctx, bs, [batch.k_cache[:, :, :hh],
                                                      batch.v_cache[:, :, :hh]])
    slots = batch.slot_mapping.cpu().numpy()[:n]
    slots2 = np.array([remap[int(s_) // bs] * bs + int(s_) % bs for s_ in slots], np.int64)
    return (batch.q.cpu()[:n, :hh].contiguous().numpy(), np.ascontiguousarray(kc),
            np.ascontiguousarray(vc), bt2, ctx,
            batch.k_new.cpu()[:n, :hh].contiguous().numpy(),
            batch.v_new.cpu()[:n, :hh].contiguous().numpy(), slots2)


def run_reference(args):
    import oracle
    batch = make_workload("cpu", seed=1)
    H, D, bs = batch.H, batch.D, batch.block_size
    ctx_all = batch.context_lens.numpy()
    budget = args.reference_budget_s / max(args.steps + args.warmup, 1)
    with one_core() as info:
        # calibrate: the oracle's cost per attended (key, head) on one sequence, one head
        one = compact_sample(batch, 1, heads=1)
        t0 = time.perf_counter()
        kc2, vc2 = oracle.kv_cache_write(one[5], one[6], one[7], one[1], one[2])
        oracle.decode(one[0], kc2, vc2, one[3], one[4], batch.scale)
        per_key_head = (time.perf_counter() - t0) / int(ctx_all[0])
        n, heads = 1, H
        if per_key_head * ctx_all[0] * H > budget:  # less than one whole sequence: fewer heads
            heads = int(max(1, min(H, budget // (per_key_head * ctx_all[0]))))
        else:
            while n < len(ctx_all) and per_key_head * H * ctx_all[:n + 1].sum() < budget:
                n += 1
        q, kc, vc, bt, ctx, kn, vn, sm = compact_sample(batch, n, heads)

        def one_step():
            kc2, vc2 = oracle.kv_cache_write(kn, vn, sm, kc, vc)
            oracle.decode(q, kc2, vc2, bt, ctx, batch.scale)

        for _ in range(args.warmup):
            one_step()
        ts = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            one_step()
            ts.append(time.perf_counter() - t0)
    byts = decode_bytes(ctx, n, heads, D, bs) + write_bytes(n, heads, D)
    secs = sum(ts)
    value = byts * args.steps / secs / 1e9
    sample = (f"cache write of {n} new token(s) + decode of the first {n} of {len(ctx_all)} "
              f"sequences, {heads} of {H} heads ({int(ctx.sum())} keys) per step, on a pool "
              "of only their blocks; fp64, one thread pinned to one core")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(batch),
        "cpu_baseline": cpu_line(value, "GB/s", secs, sample, info, None),
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
def aggregate_ranks(timed_s, e2e_s, step_bytes, world, device):
    """Whole-job numbers of N independent replicas: the slowest rank's times
    (max over ranks) and the bytes of all ranks (sum).  Host-side only; the
    data path has no collective."""
    if world <= 1:
        return timed_s, e2e_s, float(step_bytes)
    t = torch.tensor([timed_s, e2e_s], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    b = torch.tensor([float(step_bytes)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(b)
    timed_s, e2e_s = t.tolist()
    return timed_s, e2e_s, b.item()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0,
                    help="oracle seconds for the headline step's CPU baseline")
    ap.add_argument("--workload-cpu-budget-s", type=float, default=4.0,
                    help="oracle seconds per other workload's CPU baseline")
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="omit the other workloads from the default line")
    ap.add_argument("--block-size", type=int, default=16,
                    help="physical block size of the synthetic pools (16 or 32)")
    ap.add_argument("--clock-window-s", type=float, default=0.5,
                    help="seconds of back-to-back steps after each timed region, sampled for "
                         "the clock record (0: none)")
    ap.add_argument("--context-len", type=int, default=1 << 20,
                    help="tokens of the long-context sequence (a smaller one for captures)")
    ap.add_argument("--workload", default="llama13b_decode",
                    choices=("llama13b_decode",) + WORKLOADS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    from paged_kv_cache_172_gb300 import build_lib
    build_lib.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    cpu_budget = 0.0 if args.no_cpu_baseline else args.workload_cpu_budget_s
    if args.workload != "llama13b_decode":  # one workload on its own line
        sampler = ClockSampler(dev).start()
        try:
            entry = measure_workload(args.workload, args, dev, sampler, peaks, cpu_budget)
        finally:
            sampler.stop()
        entry.update({"n_gpus": 1, "higher_is_better": True,
                      "dtype": "f16 storage, f32 accumulate", "data": "synthetic (seeded fp16 "
                      "N(0,1))", "config": {"workload": entry.pop("workload")}})
        print(json.dumps(entry))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    sampler = ClockSampler(dev).start()
    try:
        res = run_gpu(args, rank, world, local_rank)
        K = args.steps
        total_s = res["step_ms"] * K / 1e3
        step_bytes = res["step_bytes"]
        e2e_ms, h2d, d2h, wall_ms, wall_med = res["e2e"][True]
        total_s, e2e_s, all_bytes = aggregate_ranks(total_s, e2e_ms * K / 1e3, step_bytes, world,
                                                    "cuda")
        wl = {}
        if rank == 0 and world == 1 and not args.no_workloads:
            for name in WORKLOADS:
                wl[name] = measure_workload(name, args, dev, sampler, peaks, cpu_budget)
    finally:
        sampler.stop()
    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    (peak, peak_kind), _ = peaks
    value = all_bytes * K / total_s / 1e9
    # the step is one pa_decode_append call: its algorithmic bytes over its duration
    achieved = step_bytes / (res["step_ms"] / 1e3) / 1e9
    batch = res["batch"]
    staged = res["e2e"][False]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_s / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 storage, f32 accumulate",
        "data": "synthetic (seeded fp16 N(0,1))",
        "config": workload_config(batch),
        "launch": {"partition_tokens": res["partition_tokens"], "num_parts": res["num_parts"],
                   "l2": "flushed before every timed step (512 MB read, untimed)"},
        "frac_of_nominal_8tbs": value / NOMINAL_HBM_GBS,
        f"frac_of_{peak_kind}_hbm": value / peak,
        "attended_tokens_per_s": res["tokens"] * world / (res["step_ms"] / 1e3),
        "step_ms_median": res["step_ms_median"],
        "sustained": res["sustained"],
        "two_launch_path": {"ms_per_step": res["unfused_ms"], "write_ms": res["write_ms"],
                            "decode_ms": res["decode_ms"],
                            "decode_GBs": res["decode_bytes"] / (res["decode_ms"] / 1e3) / 1e9},
        "roofline": {"bound": "hbm",
                     "kernel": "pa_decode_append (partition kernel with the fused cache write, "
                               "+ combine kernel)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic_for("llama13b_decode", args.block_size),
                     "traffic_kernel": "partition_kernel", "algorithmic_bytes": step_bytes},
        "e2e": {"value": all_bytes * K / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s / K * 1e3,
                "path": "DecodeSession.step_from_host: the kernels load q, k_new, v_new, "
                        "context_lens and block_tables from pinned host memory over the "
                        "host link and store out there (no copy call)",
                "host_wall_ms_per_step": wall_ms, "host_wall_ms_median": wall_med,
                "host_wall_GBs": step_bytes / (wall_ms / 1e3) / 1e9,
                "staged_ms_per_step": staged[0], "staged_h2d_bytes_per_step": staged[1],
                "staged_host_wall_ms_per_step": staged[3]},
        "gpu_launches": res["launches"],
        "clocks": sampler.summary(res["windows"]),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batch, args.cpu_budget_s)
    if wl:
        line["workloads"] = wl
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
