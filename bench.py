"""Benchmark of the paged-decode hot path on GB300.

One step = the cache write of the batch's 38 new tokens fused into paged
decode (pa_decode_append: split partitions + log-sum-exp combine; the
two-launch path pa_kv_cache_write + pa_decode is timed beside it) over the
LLaMA-13B-shaped batch: 38
sequences, 40 heads, head_dim 128, block_size 16, context lengths uniform in
[128, 2048], fp16 N(0,1) synthetic data.  The metric is algorithmic HBM
GB/s (K+V rows attended + q + out + table/length reads + the cache write's
read and write), plus attended tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Multi-GPU (torchrun): every rank runs its own independent batch (decode
sequences are independent; no collective on the data path); value = bytes
of all ranks / max-over-ranks time, scaling "weak".
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (rank 0 only).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged-decode KV HBM GB/s (% of ~8 TB/s) and attended tokens/s, 1×GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the decode
# partition kernel (the dominant kernel) from an ncu capture of this bench's
# 38-sequence batch, keyed by the hash of the decode source it was taken on;
# null once the source changes.
# (Later keys: the same partition kernel; the file changed elsewhere -- the
# combine kernel, the box-size rule shared with the maps.)
DECODE_TRAFFIC = {"9567fb4ba38dcdb0": 853235456 + 5994752,
                  "ca9f4bc9ad9c7b93": 853235456 + 5994752,
                  "c9210cf186a5438a": 853235456 + 5994752}
# The same for one launch of the chunked-prefill kernel (8 x 512 queries on
# 3,584 cached tokens, block size 16), keyed by the hash of the prefill source.
# (The second key: the same kernel with a tile-wide decision before its
# epilogue; same-box timing identical.)
PREFILL_TRAFFIC = {("167764288f8a5ffe", 16): 713364224 + 46671872,
                   ("ed8f25aa633200ea", 16): 713364224 + 46671872}


def src_hash(name):
    p = os.path.join(ROOT, "paged_kv_cache_172_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# workload and byte accounting
# ---------------------------------------------------------------------------
def decode_bytes(ctx, B, H, D, bs):
    ctx = np.asarray(ctx, dtype=np.int64)
    kv = int(ctx.sum()) * H * D * 2 * 2
    qo = 2 * B * H * D * 2
    tables = int(sum(-(-int(c) // bs) for c in ctx)) * 4 + B * 4
    return kv + qo + tables


def write_bytes(T, H, D):
    return 2 * (2 * T * H * D * 2) + T * 8


def make_workload(device, seed=1, block_size=16):
    from paged_kv_cache_172_gb300 import workloads
    return workloads.llama13b_decode(seed=seed, device=device, block_size=block_size)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def run_gpu(args, rank, world, local_rank):
    import paged_kv_cache_172_gb300 as pk
    from paged_kv_cache_172_gb300 import build_lib
    from paged_kv_cache_172_gb300.session import DecodeSession

    build_lib.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
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
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        # Read (not write) a buffer 4x the L2 size: the L2 ends up holding clean
        # lines only, so no write-back of flush data lands in the timed region.
        torch.sum(flush, dim=0, out=flush_sink)

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
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            for i in range(K):
                flush_l2()  # evict the previous step from L2 (untimed)
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the timed region")
    total_ms = sum(step_ms)

    # -- the same step as two launches (cache write, then decode), for reference
    uev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            uev[i][0].record(stream)
            write_unfused()
            uev[i][1].record(stream)
            decode_unfused()
            uev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    dec_ms = [uev[i][1].elapsed_time(uev[i][2]) for i in range(K)]
    wr_ms = [uev[i][0].elapsed_time(uev[i][1]) for i in range(K)]
    unfused_ms = [uev[i][0].elapsed_time(uev[i][2]) for i in range(K)]

    # -- end to end: host buffers, copies inside the timed region ---------------
    # Zero copy (the session's default): the kernels load every input from
    # pinned host memory and store out there.  Staged: one copy in, one out.
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
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                sess.step_from_host(host, status=status, stream=stream)
        torch.cuda.synchronize(dev)
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
        with torch.cuda.stream(stream):
            for i in range(K):
                flush_l2()
                e2e_ev[i][0].record(stream)
                sess.step_from_host(host, status=status, stream=stream)
                e2e_ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        if not torch.equal(host["out"], ref_out):
            raise RuntimeError("end-to-end output differs from the device-resident run")
        e2e[zero_copy] = (sum(a.elapsed_time(b) for a, b in e2e_ev), sess.h2d_bytes(),
                          sess.d2h_bytes())
    e2e_ms, h2d, d2h = e2e[True]

    dbytes = decode_bytes(ctx, B, H, D, bs)
    sbytes = dbytes + write_bytes(int(batch.slot_mapping.numel()), H, D)
    res = {
        "step_ms": total_ms / K, "step_ms_median": statistics.median(step_ms),
        "decode_ms": statistics.mean(dec_ms),
        "decode_ms_median": statistics.median(dec_ms), "write_ms": statistics.mean(wr_ms),
        "unfused_ms": statistics.mean(unfused_ms),
        "e2e_ms": e2e_ms / K, "e2e_staged_ms": e2e[False][0] / K,
        "e2e_staged_h2d": e2e[False][1], "step_bytes": sbytes, "decode_bytes": dbytes,
        "tokens": int(ctx.sum()), "clocks": clocks.summary(), "partition_tokens": pt,
        "num_parts": n_parts, "launches": launches_per_step * K,
        "h2d": h2d, "d2h": d2h,
        "batch": batch,
    }
    return res


def cpu_baseline(batch, budget_s):
    """Time the fp64 oracle (single thread) on a bounded sample of the
    workload: the cache write of the new tokens, then decode of the first
    sequences whose estimated cost fits ``budget_s``."""
    import oracle
    kc = batch.k_cache.cpu().numpy()
    vc = batch.v_cache.cpu().numpy()
    q = batch.q.cpu().numpy()
    bt = batch.block_tables.cpu().numpy()
    ctx = batch.context_lens.cpu().numpy()
    kn, vn = batch.k_new.cpu().numpy(), batch.v_new.cpu().numpy()
    sm = batch.slot_mapping.cpu().numpy()
    H, D, bs = batch.H, batch.D, batch.block_size
    # calibrate: one sequence
    t0 = time.perf_counter()
    oracle.decode(q[:1], kc, vc, bt[:1], ctx[:1], batch.scale)
    per_token = (time.perf_counter() - t0) / max(int(ctx[0]), 1)
    n = 1
    while n < len(ctx) and per_token * ctx[:n + 1].sum() < budget_s:
        n += 1
    t0 = time.perf_counter()
    kc2, vc2 = oracle.kv_cache_write(kn, vn, sm, kc, vc)
    oracle.decode(q[:n], kc2, vc2, bt[:n], ctx[:n], batch.scale)
    dt = time.perf_counter() - t0
    byts = decode_bytes(ctx[:n], n, H, D, bs) + write_bytes(len(sm), H, D)
    return {"value": byts / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": dt,
            "sample": f"cache write of {len(sm)} tokens + decode of the first {n} of "
                      f"{len(ctx)} sequences ({int(ctx[:n].sum())} keys x {H} heads), fp64, "
                      "single thread"}


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
    used = []
    for b in range(n):
        used.extend(int(x) for x in bt[b, :-(-int(ctx[b]) // bs)])
    uniq = sorted(set(used))
    remap = {old: new for new, old in enumerate(uniq)}
    idx = torch.as_tensor(uniq, dtype=torch.int64)
    kc = batch.k_cache.cpu()[idx][:, :, :hh].contiguous().numpy()
    vc = batch.v_cache.cpu()[idx][:, :, :hh].contiguous().numpy()
    bt2 = np.full_like(bt, -1)
    for b in range(n):
        nb = -(-int(ctx[b]) // bs)
        bt2[b, :nb] = [remap[int(x)] for x in bt[b, :nb]]
    slots = batch.slot_mapping.cpu().numpy()[:n]
    slots2 = np.array([remap[int(s_) // bs] * bs + int(s_) % bs for s_ in slots], np.int64)
    return (batch.q.cpu()[:n, :hh].contiguous().numpy(), kc, vc, bt2, ctx,
            batch.k_new.cpu()[:n, :hh].contiguous().numpy(),
            batch.v_new.cpu()[:n, :hh].contiguous().numpy(), slots2)


def run_reference(args):
    import oracle
    batch = make_workload("cpu", seed=1)
    H, D, bs = batch.H, batch.D, batch.block_size
    ctx_all = batch.context_lens.numpy()
    budget = args.reference_budget_s / max(args.steps + args.warmup, 1)
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
              "of only their blocks; fp64, one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(batch, None, "n/a (CPU)"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def workload_config(batch, pt, l2):
    ctx = batch.context_lens.cpu().numpy()
    return {"workload": f"llama13b_decode_b38: 38 seqs x 40 heads x head_dim 128, block_size "
                        f"{batch.block_size}, context_lens U[128,2048] (seed 1), pool 1.2x "
                        "need, randomly permuted blocks; step = cache write of 38 new tokens "
                        "fused into decode (pa_decode_append)",
            "B": int(batch.B), "H": int(batch.H), "head_dim": int(batch.D),
            "block_size": int(batch.block_size), "num_blocks": int(batch.num_blocks),
            "sum_context_len": int(ctx.sum()), "partition_tokens": pt, "l2": l2}


# ---------------------------------------------------------------------------
# auxiliary workloads (measurement lines for the other paged-attention cases;
# the default line above stays the 38-sequence decode)
# ---------------------------------------------------------------------------
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


def run_aux(args, name):
    import paged_kv_cache_172_gb300 as pk
    from paged_kv_cache_172_gb300 import build_lib, workloads

    build_lib.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)
    peak_hbm, hbm_kind = measured_peak()
    extra = {}
    extra_fns = {}
    if name == "prefix_sharing":
        batch = workloads.prefix_sharing(seed=2, device=dev)
        lay = batch.meta["layout"]
        ctx = lay.context_lens
        max_ctx = int(ctx.max())
        out = torch.empty_like(batch.q)
        H, D, bs = batch.H, batch.D, batch.block_size
        sg, off, seqs, pref = (torch.from_numpy(x).to(dev)
                               for x in workloads.sharing_groups(lay))
        max_prefix = int(pref.max())
        pt = max_prefix // 3  # 336: three partitions cover the 1,008 shared tokens
        phases = [
            ("block_copy", lambda: pk.pa_block_copy(batch.k_cache, batch.v_cache,
                                                    batch.copy_pairs, status=status,
                                                    stream=stream)),
            ("decode", lambda: pk.pa_decode_shared_prefix(
                batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                batch.context_lens, sg, off, seqs, pref, batch.scale, max_ctx, 8, max_prefix,
                out=out, partition_tokens=pt, status=status, stream=stream)),
        ]
        extra_fns["decode_without_sharing"] = lambda: pk.pa_decode(
            batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.context_lens,
            batch.scale, max_ctx, out=out, status=status, stream=stream)
        logical = decode_bytes(ctx, batch.B, H, D, bs)
        unique = unique_kv_bytes(lay.tables, ctx, bs, H, D) + 2 * batch.B * H * D * 2
        copy_bytes = 2 * 2 * len(lay.pairs) * bs * H * D * 2
        main, work, unit, bound = "decode", unique, "GB/s", "hbm"
        extra = {"logical_bytes": logical, "unique_bytes": unique, "copy_bytes": copy_bytes}
        desc = ("prefix_sharing_16x8: 16 prompts x 8 samples, 1024-token shared prompts, "
                "tails U[1,512], 40 heads, head_dim 128, block_size 16; step = block_copy of "
                "128 copy-on-write blocks + pa_decode_shared_prefix (groups of 8 sharing "
                "1,008 tokens, 336-token partitions); GB/s on unique bytes")
    elif name == "llama13b_decode_fp8":
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
        work = int(ctx.sum()) * H * (2 * D + 8) + 2 * batch.B * H * D * 2 + \
            int(sum(-(-int(c) // bs) for c in ctx)) * 4 + batch.B * 4
        main, unit, bound = "decode", "GB/s", "hbm"
        extra = {"fp8_algorithmic_bytes": work,
                 "fp16_equivalent_bytes": decode_bytes(ctx, batch.B, H, D, bs),
                 "write_fp8_bytes": T * H * (2 * 2 * D + 2 * D + 8)}
        desc = ("llama13b_decode_b38_fp8: the 38-sequence batch stored as e4m3 with "
                "per-(token, head) fp32 scales; step = quantizing write of 38 new tokens + "
                "pa_decode_fp8; GB/s on fp8 bytes")
    elif name == "long_context":
        batch = workloads.long_context(seed=3, device=dev, bs=args.block_size)
        n = int(batch.context_lens[0])
        out = torch.empty_like(batch.q)
        H, D, bs = batch.H, batch.D, batch.block_size
        phases = [("decode", lambda: pk.pa_decode(batch.q, batch.k_cache, batch.v_cache,
                                                  batch.block_tables, batch.context_lens,
                                                  batch.scale, n, out=out, status=status,
                                                  stream=stream))]
        work = decode_bytes([n], 1, H, D, bs)
        main, unit, bound = "decode", "GB/s", "hbm"
        desc = (f"long_context_1M: 1 sequence of 1,048,576 tokens, 40 heads, head_dim 128, "
                f"block_size {bs}, {batch.num_blocks} permuted blocks; split-KV decode")
    elif name == "chunked_prefill":
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
        main, unit, bound = "prefill", "TFLOP/s", "tensor"
        extra = {"useful_flops": work,
                 "kv_bytes": int(ctx.sum()) * H * D * 4, "q_out_bytes": 2 * batch.q.numel() * 2}
        desc = (f"chunked_prefill_8x512_on_3584: 8 sequences, 512-query chunk on 3,584 cached "
                f"tokens (context 4,096), 40 heads, head_dim 128, block_size {bs}; step = "
                "kv_cache_write of the 4,096 chunk tokens + pa_prefill_chunk")
    else:
        raise SystemExit(f"unknown workload {name}")

    def run_step(evs=None):
        for i, (_, fn) in enumerate(phases):
            if evs is not None:
                evs[i].record(stream)
            fn()
        if evs is not None:
            evs[-1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            torch.sum(flush, dim=0, out=flush_sink)
            run_step()
    torch.cuda.synchronize(dev)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
           for _ in range(K)]
    with ClockSampler(0) as clocks:
        with torch.cuda.stream(stream):
            for i in range(K):
                torch.sum(flush, dim=0, out=flush_sink)
                run_step(evs[i])
        torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x}")
    phase_ms = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, (nm, _) in enumerate(phases)}
    for nm, fn in extra_fns.items():  # alternatives timed beside the step, same flushing
        xs = []
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
            for _ in range(K):
                torch.sum(flush, dim=0, out=flush_sink)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                xs.append((e0, e1))
        torch.cuda.synchronize(dev)
        extra[f"{nm}_ms"] = statistics.mean(a.elapsed_time(b) for a, b in xs)
    step_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in evs)
    main_s = phase_ms[main] / 1e3
    if bound == "tensor":
        achieved = work / main_s / 1e12
        peak, peak_kind = 1904.1, "measured bf16 burst (fp16 dense rate equal)"
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                peak = float(json.load(f)["bf16_tflops"])
        except Exception:
            peak, peak_kind = 1900.0, "fallback"
    else:
        achieved = work / main_s / 1e9
        peak, peak_kind = peak_hbm, hbm_kind
    line = {
        "metric": f"{name} {unit}", "value": achieved, "unit": unit, "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "dtype": "f16 storage, f32 accumulate", "data": "synthetic (seeded fp16 N(0,1))",
        "config": {"workload": desc, "l2": "flushed before every timed step (512 MB read)"},
        "phase_ms": phase_ms,
        "roofline": {"bound": bound, "kernel": main, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": None},
        "clocks": clocks.summary(),
    }
    if name == "chunked_prefill":
        line["roofline"]["traffic"] = PREFILL_TRAFFIC.get((src_hash("prefill.cu"), args.block_size))
        line["roofline"]["traffic_kernel"] = "prefill_kernel"
    line.update(extra)
    if name == "prefix_sharing":
        line["logical_GBs"] = logical / main_s / 1e9
    if name == "llama13b_decode_fp8":
        line["attended_tokens_per_s"] = int(ctx.sum()) / main_s
    print(json.dumps(line))


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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--block-size", type=int, default=16,
                    help="physical block size of the synthetic pools (16 or 32)")
    ap.add_argument("--workload", default="llama13b_decode",
                    choices=["llama13b_decode", "prefix_sharing", "long_context",
                             "chunked_prefill", "llama13b_decode_fp8"])
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.workload != "llama13b_decode":
        run_aux(args, args.workload)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, rank, world, local_rank)
    K = args.steps
    total_s = res["step_ms"] * K / 1e3
    step_bytes = res["step_bytes"]
    dec_s = res["decode_ms"] / 1e3
    total_s, e2e_s, all_bytes = aggregate_ranks(total_s, res["e2e_ms"] * K / 1e3,
                                                step_bytes, world, "cuda")
    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    value = all_bytes * K / total_s / 1e9
    # the step is one pa_decode_append call: its algorithmic bytes over its duration
    achieved = step_bytes / (res["step_ms"] / 1e3) / 1e9
    key = src_hash("decode.cu")
    traffic = DECODE_TRAFFIC.get(key)
    batch = res["batch"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_s / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 storage, f32 accumulate",
        "data": "synthetic (seeded fp16 N(0,1))",
        "config": workload_config(batch, res["partition_tokens"],
                                  "flushed before every timed step (512 MB read, untimed)"),
        "frac_of_nominal_8tbs": value / NOMINAL_HBM_GBS,
        f"frac_of_{peak_kind}_hbm": value / peak,
        "attended_tokens_per_s": res["tokens"] * world / (res["step_ms"] / 1e3),
        "step_ms_median": res["step_ms_median"],
        "two_launch_path": {"ms_per_step": res["unfused_ms"], "write_ms": res["write_ms"],
                            "decode_ms": res["decode_ms"],
                            "decode_GBs": res["decode_bytes"] / dec_s / 1e9},
        "roofline": {"bound": "hbm",
                     "kernel": "pa_decode_append (partition kernel with the fused cache write, "
                               "+ combine kernel)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic, "traffic_kernel": "partition_kernel",
                     "algorithmic_bytes": step_bytes},
        "e2e": {"value": all_bytes * K / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": e2e_s / K * 1e3,
                "path": "DecodeSession.step_from_host: the kernels load q, k_new, v_new, "
                        "context_lens and block_tables from pinned host memory over the "
                        "host link and store out there (no copy call)",
                "staged_ms_per_step": res["e2e_staged_ms"],
                "staged_h2d_bytes_per_step": res["e2e_staged_h2d"]},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batch, args.cpu_budget_s)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
