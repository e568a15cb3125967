"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

# Attention tolerance for fp16 output from an fp32 accumulation against the
# fp64 oracle, unit-normal inputs: max |err| <= 5e-3 and mean |err| <= 5e-4.
MAX_ABS = 5e-3
MEAN_ABS = 5e-4


def errors(out, ref):
    got = out.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    return float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0


def assert_close(out, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    mx, mean = errors(out, ref)
    assert mx <= max_abs and mean <= mean_abs, \
        f"{what}: max|err| {mx:.3e} (<= {max_abs}), mean|err| {mean:.3e} (<= {mean_abs})"
    return mx, mean


def bits(t):
    """Device or host fp16 tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().numpy().view(np.uint16)


def to_dev(batch, dev, names=("q", "k_cache", "v_cache", "block_tables", "context_lens",
                              "k_new", "v_new", "slot_mapping", "copy_pairs")):
    out = {}
    for n in names:
        t = getattr(batch, n)
        if t is not None:
            out[n] = t.to(dev)
    return out


def zero_status(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def spiked_decode_batch(D, bs, seed):
    """Scores with jumps far past any rescale margin, spread over partitions:
    queries u + noise (u = ones), chosen keys a * u (about a * D above the
    rest).  Sequence 0: the spike at the last key; 1: spikes of growing size in
    three partitions; 2: the largest score at key 0; 3: no spike; 4: every
    eighth key far below the rest."""
    ctx = [1024, 1024, 1024, 700, 900]
    from paged_kv_cache_172_gb300 import workloads
    batch = workloads.random_decode(len(ctx), 2, D, bs, ctx, seed=seed, device="cpu")
    g = torch.Generator().manual_seed(seed)
    batch.q = (1.0 + 0.25 * torch.randn(batch.q.shape, generator=g)).half()
    per_nat = 1.0 / (D * batch.scale)
    marks = {0: [(ctx[0] - 1, 45)], 1: [(100, 15), (400, 35), (700, 60)], 2: [(0, 60)],
             4: [(p, -40) for p in range(0, ctx[4], 8)]}
    for b, ms in marks.items():
        for pos, nats in ms:
            blk = int(batch.block_tables[b, pos // bs])
            batch.k_cache[blk, pos % bs] = torch.full((2, D), nats * per_nat).half()
    return batch

