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
