"""pa_decode_static: decode attention for callers that cannot allocate.

Some callers of this library cannot allocate device memory for a call (a
runtime that gave the whole device heap to its own pool, a plugin that must
not allocate outside its host engine, a loop that cannot pay for
cudaMalloc's implicit synchronisation).  pa_decode_static serves them: it
takes pa_decode's arguments minus the workspace and keeps the split-KV
scratch in a fixed array inside the library.  This test calls it through
the C ABI and checks that two calls in a row match pa_decode (which uses a
caller-owned workspace) within the attention tolerance, the second call
running on fresh inputs over the scratch the first one left behind; and
that a plan larger than the fixed array is refused.

The file name sorts last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def call_static(g, batch, max_ctx, pt, out, status):
    lib = pk.lib()
    NB, bs, H, D = g["k_cache"].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return lib.pa_decode_static(_p(g["q"]), _p(g["k_cache"]), _p(g["v_cache"]),
                                _p(g["block_tables"]), _p(g["context_lens"]), g["q"].shape[0],
                                H, D, bs, NB, g["block_tables"].shape[1], max_ctx, pt,
                                ctypes.c_float(batch.scale), _p(out), _p(status), stream)


def test_static_scratch_matches_workspace_path_twice():
    ctx = [2048, 1, 700, 1500, 129, 0, 33, 1024]
    max_ctx = 2048
    pt = 128  # 16 partitions: the scratch array is used
    need = pk.pa_decode_workspace_size(len(ctx), 8, 128, 16, max_ctx, pt)
    assert 0 < need <= pk._lib.PA_DECODE_STATIC_SCRATCH_BYTES
    for seed in (31, 32):  # two calls in a row, the second over stale scratch
        batch = workloads.random_decode(len(ctx), 8, 128, 16, ctx, seed=seed, device=DEV)
        g = {k: getattr(batch, k) for k in ("q", "k_cache", "v_cache", "block_tables",
                                            "context_lens")}
        ref = pk.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                           g["context_lens"], batch.scale, max_ctx, partition_tokens=pt)
        out = torch.full_like(g["q"], float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = call_static(g, batch, max_ctx, pt, out, status)
        assert rc == pk.PA_OK, pk.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        err = (out.float() - ref.float()).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
        assert torch.all(out[5] == 0)  # empty sequence


def test_static_single_partition_and_empty_batch():
    # One partition (partition_tokens >= max_context_len): no scratch is
    # needed and the array is not touched; then a batch whose contexts are
    # all 0 (max_context_len 0 is planned as 1).  Both against pa_decode.
    for ctx, max_ctx, pt in (([300, 1, 512, 77], 512, 512), ([0, 0, 0], 0, 0)):
        batch = workloads.random_decode(len(ctx), 4, 128, 16, ctx, seed=41, device=DEV,
                                        extra_blocks=2)
        g = {k: getattr(batch, k) for k in ("q", "k_cache", "v_cache", "block_tables",
                                            "context_lens")}
        assert pk.pa_decode_workspace_size(len(ctx), 4, 128, 16, max(max_ctx, 1), pt) == 0
        ref = pk.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                           g["context_lens"], batch.scale, max_ctx, partition_tokens=pt)
        out = torch.full_like(g["q"], float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = call_static(g, batch, max_ctx, pt, out, status)
        assert rc == pk.PA_OK, pk.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref)  # same kernel, same plan: identical bits
        if max_ctx == 0:
            assert torch.all(out == 0)


def test_static_scratch_rejects_oversized_plan():
    # 64 sequences x 40 heads x 64 partitions of 32 tokens x (128 + 2) floats
    # is 85 MB of scratch, more than the fixed array holds: refused before launch.
    B, H, D, bs, maxb = 64, 40, 128, 16, 128
    assert pk.pa_decode_workspace_size(B, H, D, bs, 2048, 32) > \
        pk._lib.PA_DECODE_STATIC_SCRATCH_BYTES
    g = {"q": torch.zeros((B, H, D), dtype=torch.float16, device=DEV),
         "k_cache": torch.zeros((4, bs, H, D), dtype=torch.float16, device=DEV),
         "v_cache": torch.zeros((4, bs, H, D), dtype=torch.float16, device=DEV),
         "block_tables": torch.zeros((B, maxb), dtype=torch.int32, device=DEV),
         "context_lens": torch.ones(B, dtype=torch.int32, device=DEV)}

    class _Scale:
        scale = 0.1

    out = torch.empty_like(g["q"])
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert call_static(g, _Scale, 2048, 32, out, status) == pk.PA_ERR_WORKSPACE
