"""DecodeSession: per-step inputs from pinned host buffers, either read by
the kernel in place (zero copy: only context lengths and tables are copied)
or staged by one packed host->device copy with one device->host copy of the
output.  Its result must equal the device-resident call bit for bit (output
and cache write), and the oracle's cache write + decode."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from paged_kv_cache_172_gb300.session import DecodeSession
from pk_testutil import assert_close, bits, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


@pytest.mark.parametrize("zero_copy", [True, False])
@pytest.mark.parametrize("bs,D", [(16, 128), (32, 128), (16, 64)])
def test_session_matches_device_call_and_oracle(bs, D, zero_copy):
    ctx = [1, bs + 1, 3 * bs, 517, 2048]
    batch = workloads.random_decode(len(ctx), 6, D, bs, ctx, seed=90 + bs + D, device="cpu",
                                    new_tokens=True)
    max_ctx = max(ctx)
    # device-resident call on one copy of the pool
    g = {k: getattr(batch, k).to(DEV) for k in ("q", "k_cache", "v_cache", "block_tables",
                                                "context_lens", "k_new", "v_new")}
    status = zero_status(DEV)
    out_dev = pk.pa_decode_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"],
                                  g["block_tables"], g["context_lens"], batch.scale, max_ctx,
                                  status=status)
    # the session on another copy, inputs from pinned host buffers
    kc2, vc2 = batch.k_cache.to(DEV), batch.v_cache.to(DEV)
    sess = DecodeSession(kc2, vc2, len(ctx), batch.block_tables.shape[1], max_ctx, batch.scale,
                         zero_copy=zero_copy)
    host = sess.host_buffers()
    for name in ("q", "k_new", "v_new", "context_lens", "block_tables"):
        host[name].copy_(getattr(batch, name))
    status2 = zero_status(DEV)
    for _ in range(2):  # the second step rewrites the same slots with the same values
        sess.step_from_host(host, status=status2)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(status2.item()) == 0
    assert torch.equal(host["out"], out_dev.cpu())
    assert torch.equal(kc2, g["k_cache"]) and torch.equal(vc2, g["v_cache"])
    assert sess.h2d_bytes() >= sum(getattr(batch, n).numel() * getattr(batch, n).element_size()
                                   for n in ("q", "k_new", "v_new", "context_lens", "block_tables"))
    assert sess.h2d_bytes() <= sess._stage_bytes
    kc, vc = oracle.kv_cache_write(batch.k_new.numpy(), batch.v_new.numpy(),
                                   batch.slot_mapping.numpy(), batch.k_cache.numpy(),
                                   batch.v_cache.numpy())
    assert np.array_equal(bits(kc2), kc) and np.array_equal(bits(vc2), vc)
    ref = oracle.decode(batch.q.numpy(), kc, vc, batch.block_tables.numpy(),
                        batch.context_lens.numpy(), batch.scale)
    assert_close(host["out"], ref, what=f"session bs={bs} D={D}")


def test_session_rejects_foreign_host_buffers():
    batch = workloads.random_decode(2, 2, 64, 16, [5, 9], seed=7, device="cpu", new_tokens=True)
    sess = DecodeSession(batch.k_cache.to(DEV), batch.v_cache.to(DEV), 2,
                         batch.block_tables.shape[1], 9, batch.scale)
    with pytest.raises(ValueError):
        sess.step_from_host({"q": batch.q.pin_memory()})


def test_host_device_pointer():
    pinned = torch.zeros(1000, dtype=torch.float16).pin_memory()
    d = pk.host_device_pointer(pinned)
    assert d  # unified addressing: the host address itself
    assert pk.host_device_pointer(pinned[8:]) == d + 16  # inside the allocation
    with pytest.raises(pk.PagedKVError):
        pk.host_device_pointer(torch.zeros(1000, dtype=torch.float16))  # pageable
    with pytest.raises(TypeError):
        pk.host_device_pointer(torch.zeros(4, device=DEV))


@pytest.mark.parametrize("tables_on_host", [False, True])
@pytest.mark.parametrize("bs", [16, 32])
def test_decode_with_host_inputs_and_output(bs, tables_on_host):
    """q and out (and the tables and lengths) in pinned host memory, read
    and written by the kernels in place, give the device-resident result bit
    for bit, split-KV included."""
    ctx = [1, 300, 1200, 2048]
    batch = workloads.random_decode(len(ctx), 8, 128, bs, ctx, seed=200 + bs, device=DEV)
    ref = pk.pa_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                       batch.context_lens, batch.scale, max(ctx), partition_tokens=256)
    q_h = batch.q.cpu().pin_memory()
    out_h = torch.full(q_h.shape, float("nan"), dtype=torch.float16).pin_memory()
    bt, cl = batch.block_tables, batch.context_lens
    if tables_on_host:
        bt, cl = bt.cpu().pin_memory(), cl.cpu().pin_memory()
    status = zero_status(DEV)
    pk.pa_decode(q_h, batch.k_cache, batch.v_cache, bt, cl, batch.scale, max(ctx), out=out_h,
                 partition_tokens=256, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out_h, ref.cpu())
