"""Two host threads drive the library at once, each on its own CUDA stream.

The kernels' one-time launch setup (the dynamic shared-memory limit of each
kernel, the SM count behind the prefill split plan) is kept per device and
is safe to reach from several threads.  The check runs in a fresh child
process, so that the two threads' very first decode, prefill and append
launches race on that setup; every output is compared with the fp64 oracle.
"""
import os
import subprocess
import sys
import threading

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _thread_inputs(seed):
    from paged_kv_cache_172_gb300 import workloads
    dec = workloads.random_decode(5, 4, 128, 16, [700, 1, 333, 64, 1200], seed=seed,
                                  device="cpu", new_tokens=True)
    pre = workloads.random_prefill(2, 3, 128, 16, 200, [640, 200], seed=seed + 1, device="cpu",
                                   write_chunk=False)
    return dec, pre


def _oracle_refs(dec, pre):
    import oracle
    ref_dec = oracle.decode(dec.q.numpy(), dec.k_cache.numpy(), dec.v_cache.numpy(),
                            dec.block_tables.numpy(), dec.context_lens.numpy(), dec.scale)
    kc, vc = oracle.kv_cache_write(dec.k_new.numpy(), dec.v_new.numpy(),
                                   dec.slot_mapping.numpy(), dec.k_cache.numpy(),
                                   dec.v_cache.numpy())
    ref_app = oracle.decode(dec.q.numpy(), kc, vc, dec.block_tables.numpy(),
                            dec.context_lens.numpy(), dec.scale)
    ref_pre = oracle.prefill(pre.q.numpy(), pre.k_cache.numpy(), pre.v_cache.numpy(),
                             pre.block_tables.numpy(), pre.context_lens.numpy(), pre.scale)
    return ref_dec, ref_app, ref_pre


def child():
    """Runs in a fresh process: two threads, first launches concurrent."""
    import torch
    import paged_kv_cache_172_gb300 as pk
    from pk_testutil import MAX_ABS, MEAN_ABS, errors

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cases = [_thread_inputs(100 + 10 * t) for t in range(2)]
    refs = [_oracle_refs(*c) for c in cases]
    start = threading.Barrier(2)
    results, failures = [None, None], []

    def work(t):
        try:
            torch.cuda.set_device(dev)
            dec, pre = cases[t]
            d = {k: getattr(dec, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_tables",
                                                      "context_lens", "k_new", "v_new")}
            p = {k: getattr(pre, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_tables",
                                                      "context_lens")}
            stream = torch.cuda.Stream(dev)
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            torch.cuda.synchronize(dev)
            start.wait()  # both threads make their first launches together
            with torch.cuda.stream(stream):
                o_dec = pk.pa_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                     d["context_lens"], dec.scale, 1200, status=status,
                                     stream=stream)
                o_pre = pk.pa_prefill_chunk(p["q"], p["k_cache"], p["v_cache"],
                                            p["block_tables"], p["context_lens"], pre.scale,
                                            status=status, stream=stream)
                o_app = pk.pa_decode_append(d["q"], d["k_new"], d["v_new"], d["k_cache"],
                                            d["v_cache"], d["block_tables"], d["context_lens"],
                                            dec.scale, 1200, status=status, stream=stream)
            stream.synchronize()
            results[t] = (o_dec.cpu(), o_app.cpu(), o_pre.cpu(), int(status.item()))
        except Exception as e:  # reported by the main thread
            failures.append(f"thread {t}: {e!r}")

    threads = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if failures:
        raise SystemExit("; ".join(failures))
    for t in range(2):
        o_dec, o_app, o_pre, st = results[t]
        assert st == 0, f"thread {t}: device status {st:#x}"
        for name, out, ref in (("decode", o_dec, refs[t][0]), ("append", o_app, refs[t][1]),
                               ("prefill", o_pre, refs[t][2])):
            mx, mean = errors(out, ref)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, \
                f"thread {t} {name}: max {mx:.3e} mean {mean:.3e}"
    print("threads ok")


@pytest.mark.gpu
def test_two_threads_first_launches_match_oracle():
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, HERE, env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "child"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


if __name__ == "__main__" and len(sys.argv) > 1 and sys.argv[1] == "child":
    for p in (ROOT, HERE):
        if p not in sys.path:
            sys.path.insert(0, p)
    child()
