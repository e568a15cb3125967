"""A bounded device wait that can never finish gives up, reports
PA_DEV_TIMEOUT in the status word, and lets the kernel return.

The kernels wait on mbarriers with a limit (about one second of SM clock in
the product library).  A test build of the library (PK_TEST_HOOKS, limit
10,000 cycles) adds one tiny kernel whose threads wait, through the same
helper, on an mbarrier that nothing arrives on and no copy completes on; no
asynchronous copy is in flight, so giving up leaves nothing behind.  Nothing
here faults, traps or hangs the GPU: the wait ends by its own limit.
"""
import ctypes
import os

import pytest
import torch

import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import build_lib

DEV = torch.device("cuda:0")
FLAGS = ("-DPK_TEST_HOOKS", "-DPK_WAIT_LIMIT_CYCLES=10000")
HOOK_LIB = os.path.join(build_lib.OBJ_DIR, "libpagedkv_testhooks.so")


def hook_lib():
    path = build_lib.build(extra_flags=FLAGS, out=HOOK_LIB, sources=["test_hooks.cu"])
    lib = ctypes.CDLL(path)
    lib.pk_test_wait_limit_cycles.restype = ctypes.c_longlong
    lib.pk_test_wait_gives_up.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_void_p]
    lib.pk_test_wait_gives_up.restype = ctypes.c_int
    return lib


def test_product_library_has_no_test_hooks():
    build_lib.build()
    raw = ctypes.CDLL(pk.LIB_PATH)
    assert not hasattr(raw, "pk_test_wait_gives_up")
    assert not hasattr(raw, "pk_test_wait_limit_cycles")


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_reports_timeout():
    lib = hook_lib()
    assert lib.pk_test_wait_limit_cycles() == 10000
    torch.cuda.set_device(DEV)
    for threads in (32, 128):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        gave_up = torch.zeros(1, dtype=torch.int32, device=DEV)
        stream = torch.cuda.current_stream(DEV)
        rc = lib.pk_test_wait_gives_up(ctypes.c_void_p(status.data_ptr()),
                                       ctypes.c_void_p(gave_up.data_ptr()), threads,
                                       ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()  # the kernel returned
        assert int(status.item()) & pk.PA_DEV_TIMEOUT
        assert int(gave_up.item()) == threads
    # the context is still usable: an ordinary library call afterwards works
    k = torch.randn((4, 8, 64), device=DEV).half()
    v = torch.randn((4, 8, 64), device=DEV).half()
    slots = torch.tensor([5, 0, 7, 2], dtype=torch.int64, device=DEV)
    kc = torch.zeros((2, 4, 8, 64), dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk.pa_kv_cache_write(k, v, slots, kc, vc, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(kc.view(8, 8, 64)[slots], k) and torch.equal(vc.view(8, 8, 64)[slots], v)
