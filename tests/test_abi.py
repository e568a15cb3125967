"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument validation returns the documented codes without touching a GPU."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import build_lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return pk.lib()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(pk.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(pk.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} missing from libpagedkv.so"


def test_status_strings(lib):
    for code in range(5):
        assert pk.status_string(code).startswith(
            ["PA_OK", "PA_ERR_INVALID", "PA_ERR_UNSUPPORTED", "PA_ERR_WORKSPACE",
             "PA_ERR_CUDA"][code])
    assert lib.pa_version() >= 100


NULL = None


def decode_rc(lib, **kw):
    args = dict(q=0x1000, k=0x1000, v=0x1000, bt=0x1000, cl=0x1000, B=2, H=4, D=128, bs=16,
                nb=8, maxb=4, maxctx=64, pt=0, scale=0.1, out=0x1000, ws=NULL, wsb=0,
                status=NULL)
    args.update(kw)
    a = args
    return lib.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"], a["H"], a["D"],
                         a["bs"], a["nb"], a["maxb"], a["maxctx"], a["pt"], a["scale"],
                         a["out"], a["ws"], a["wsb"], a["status"], NULL)


def test_decode_validation(lib):
    assert decode_rc(lib, D=96) == pk.PA_ERR_UNSUPPORTED
    assert decode_rc(lib, bs=12) == pk.PA_ERR_UNSUPPORTED
    assert decode_rc(lib, B=-1) == pk.PA_ERR_INVALID
    assert decode_rc(lib, B=0) == pk.PA_OK  # empty batch: nothing to do
    assert decode_rc(lib, q=NULL) == pk.PA_ERR_INVALID
    assert decode_rc(lib, out=0x1008) == pk.PA_ERR_INVALID  # not 16-byte aligned
    assert decode_rc(lib, nb=0) == pk.PA_ERR_INVALID
    assert decode_rc(lib, maxctx=65) == pk.PA_ERR_INVALID  # beyond table capacity
    assert decode_rc(lib, pt=24) == pk.PA_ERR_INVALID  # not a block multiple
    assert decode_rc(lib, pt=32 * 16 + 16) == pk.PA_ERR_INVALID  # > 32 blocks
    assert decode_rc(lib, scale=float("nan")) == pk.PA_ERR_INVALID
    # a split plan needs workspace
    assert decode_rc(lib, pt=16) == pk.PA_ERR_WORKSPACE
    assert decode_rc(lib, pt=16, ws=0x1000, wsb=16) == pk.PA_ERR_WORKSPACE


def static_rc(lib, **kw):
    a = dict(q=0x1000, k=0x1000, v=0x1000, bt=0x1000, cl=0x1000, B=64, H=40, D=128, bs=16,
             nb=8, maxb=128, maxctx=2048, pt=32, scale=0.1, out=0x1000, status=NULL)
    a.update(kw)
    return lib.pa_decode_static(a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"], a["H"],
                                a["D"], a["bs"], a["nb"], a["maxb"], a["maxctx"], a["pt"],
                                a["scale"], a["out"], a["status"], NULL)


def test_decode_static_validation_matches_decode(lib):
    # 64 x 40 x 64 partitions: far more scratch than the fixed array holds.
    assert pk.pa_decode_workspace_size(64, 40, 128, 16, 2048, 32) > \
        pk._lib.PA_DECODE_STATIC_SCRATCH_BYTES
    assert static_rc(lib) == pk.PA_ERR_WORKSPACE
    # An argument error gets pa_decode's code even when the plan is oversized.
    assert static_rc(lib, D=256) == pk.PA_ERR_UNSUPPORTED
    assert static_rc(lib, bs=12, pt=36) == pk.PA_ERR_UNSUPPORTED
    assert static_rc(lib, pt=24) == pk.PA_ERR_INVALID  # not a block multiple
    assert static_rc(lib, q=NULL) == pk.PA_ERR_INVALID
    assert static_rc(lib, maxctx=4096) == pk.PA_ERR_INVALID  # beyond table capacity
    assert static_rc(lib, scale=float("inf")) == pk.PA_ERR_INVALID
    assert static_rc(lib, B=0) == pk.PA_OK


def test_workspace_plan(lib):
    # 4 partitions of 16 tokens for max context 64, per (b, h): D + 2 floats
    assert pk.pa_decode_workspace_size(2, 4, 128, 16, 64, 16) == 2 * 4 * 4 * 130 * 4
    assert pk.pa_decode_workspace_size(2, 4, 128, 16, 64, 64) == 0  # one partition
    for B, H, bs, ctx in [(38, 40, 16, 2048), (1, 40, 16, 1 << 20), (4, 4, 4, 9),
                          (128, 40, 16, 1536), (1, 1, 32, 5)]:
        pt = pk.pa_decode_partition_tokens(B, H, bs, ctx)
        assert pt % bs == 0 and bs * 8 <= pt <= bs * 32
        assert (ctx + pt - 1) // pt <= 65535


def test_copy_validation(lib):
    assert lib.pa_kv_cache_write(0x1000, 0x1000, 0x1000, 4, 4, 96, 16, 8, 0x1000, 0x1000,
                                 NULL, NULL) == pk.PA_ERR_UNSUPPORTED
    assert lib.pa_kv_cache_write(0x1000, 0x1000, 0x1000, 0, 4, 128, 16, 8, 0x1000, 0x1000,
                                 NULL, NULL) == pk.PA_OK
    assert lib.pa_kv_cache_write(NULL, 0x1000, 0x1000, 4, 4, 128, 16, 8, 0x1000, 0x1000,
                                 NULL, NULL) == pk.PA_ERR_INVALID
    assert lib.pa_block_copy(0x1000, 0x1000, 0x1000, -1, 4, 128, 16, 8, NULL,
                             NULL) == pk.PA_ERR_INVALID
    assert lib.pa_block_copy(0x1000, 0x1004, 0x1000, 3, 4, 128, 16, 8, NULL,
                             NULL) == pk.PA_ERR_INVALID
    assert lib.pa_block_copy(0x1000, 0x1000, 0x1000, 0, 4, 128, 16, 8, NULL,
                             NULL) == pk.PA_OK
    p = 0x1000  # any 16-byte aligned address: these calls return before touching memory
    w8 = lambda T=4, H=4, D=128, k=p: lib.pa_kv_cache_write_fp8(k, p, p, T, H, D, 16, 8, p, p, p,
                                                                 p, NULL, NULL)
    assert w8(H=65536) == pk.PA_ERR_INVALID  # one grid row per eight heads
    assert w8(H=0) == pk.PA_ERR_INVALID
    assert w8(D=96) == pk.PA_ERR_UNSUPPORTED
    assert w8(T=0) == pk.PA_OK
    assert w8(k=NULL) == pk.PA_ERR_INVALID


def test_prefill_validation(lib):
    for D, bs in ((96, 16), (256, 16), (128, 12), (64, 64)):  # no kernel for these
        rc = lib.pa_prefill_chunk(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 2, 4, 8, D, bs, 8, 4,
                                  0.1, 0x1000, NULL, 0, NULL, NULL)
        assert rc == pk.PA_ERR_UNSUPPORTED, (D, bs)
    rc = lib.pa_prefill_chunk(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, -2, 4, 8, 128, 16, 8, 4,
                              0.1, 0x1000, NULL, 0, NULL, NULL)
    assert rc == pk.PA_ERR_INVALID
    for bad_scale in (0.0, -0.5, float("inf")):  # the prefill kernel needs scale > 0
        rc = lib.pa_prefill_chunk(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 2, 4, 8, 128, 16, 8,
                                  4, bad_scale, 0x1000, NULL, 0, NULL, NULL)
        assert rc == pk.PA_ERR_INVALID
    # chunks of different lengths: q_lens is required; otherwise as pa_prefill_chunk
    rc = lib.pa_prefill_chunk_varlen(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, NULL, 2, 4, 8, 128,
                                     16, 8, 4, 0.1, 0x1000, NULL, 0, NULL, NULL)
    assert rc == pk.PA_ERR_INVALID
    rc = lib.pa_prefill_chunk_varlen(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 2, 4, 8, 96,
                                     16, 8, 4, 0.1, 0x1000, NULL, 0, NULL, NULL)
    assert rc == pk.PA_ERR_UNSUPPORTED
    rc = lib.pa_prefill_chunk_varlen(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, NULL, 0, 4, 8, 128,
                                     16, 8, 4, 0.1, 0x1000, NULL, 0, NULL, NULL)
    assert rc == pk.PA_OK  # nothing to do


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        pk.pa_decode(q, q.view(1, 1, 1, 64), q.view(1, 1, 1, 64),
                     torch.zeros(1, 1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                     0.1, max_context_len=1)


def test_host_device_pointer_rejects_null_without_cuda(lib):
    # NULL arguments are refused before any CUDA call
    out = ctypes.c_void_p(0x1234)
    assert lib.pa_host_device_pointer(NULL, ctypes.byref(out)) == pk.PA_ERR_INVALID
    assert out.value is None
    assert lib.pa_host_device_pointer(ctypes.c_void_p(0x1000), NULL) == pk.PA_ERR_INVALID
