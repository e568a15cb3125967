"""Pins of the fp64 oracle to facts fixed outside the oracle itself.

Every ``check_*`` takes the oracle library handle so that the mutation tests
at the bottom can run the same checks against copies of the oracle with a
planted mistake, and show that each plausible mistake fails at least one pin.

Pins used:
  * IEEE-754 binary16 bit patterns with known values, and numpy's own
    float16 -> float64 conversion over all 65,536 patterns;
  * the worked examples of the study notes "DataWhale组队学习笔记--llm-algo-leetcode(五)"
    ("代码实现" test: allocation counts, the gathered shape and fill values);
  * closed forms: with q = 0 every key gets the same weight, so the output is
    the mean of the visible values (15/9 and 36/5 for the notes' fill
    patterns); one key gives that key's value; V = 1 gives 1; two keys give
    the logistic weight sigma(s0 - s1);
  * a textbook dense attention (numpy matrix form) on a contiguous copy
    built with numpy fancy indexing, for decode and for the masked chunk;
  * invariance of the output under any relabelling of physical blocks
    ("transparent to the model", notes section 3);
  * copy semantics of the cache write and block copy against numpy indexing.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import build as obuild
from oracle.allocator import BlockAllocator, OutOfBlocks, Sequence_

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


# ----------------------------------------------------------------------------
# helpers (numpy, independent of the C oracle)
# ----------------------------------------------------------------------------
def rand16(rng, shape):
    return rng.standard_normal(shape).astype(np.float16)


def paged_case(rng, B, H, D, bs, ctx, spare=3):
    need = sum(-(-c // bs) for c in ctx)
    nb = need + spare
    perm = rng.permutation(nb)
    maxb = max(1, max(-(-c // bs) for c in ctx))
    tables = np.full((B, maxb), -1, np.int32)
    pos = 0
    for b, c in enumerate(ctx):
        n = -(-c // bs)
        tables[b, :n] = perm[pos:pos + n]
        pos += n
    k = rand16(rng, (nb, bs, H, D))
    v = rand16(rng, (nb, bs, H, D))
    return k, v, tables, np.asarray(ctx, np.int32)


def contiguous(pool, table, n, h):
    """numpy fancy-index gather of logical keys 0..n-1 of head h."""
    j = np.arange(n)
    blk = np.asarray(table)[j // pool.shape[1]]
    return pool[blk, j % pool.shape[1], h, :].astype(np.float64)


def dense_attention(q, K, V, scale, mask=None):
    """Textbook softmax(scale * q K^T) V in matrix form (float64)."""
    S = scale * (q @ K.T)
    if mask is not None:
        S = np.where(mask, S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P = P / P.sum(axis=1, keepdims=True)
    return P @ V


# ----------------------------------------------------------------------------
# pins as reusable checks
# ----------------------------------------------------------------------------
KNOWN_HALF = {
    0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
    0x03FF: 1023 * 2.0 ** -24, 0x0400: 2.0 ** -14, 0x3555: 0.333251953125,
    0x3BFF: 1.0 - 2.0 ** -11, 0x4248: 3.140625, 0x0000: 0.0,
}


def check_half_known(lib):
    for bits, val in KNOWN_HALF.items():
        assert oracle.half_to_double(bits, lib=lib) == val, hex(bits)
    z = oracle.half_to_double(0x8000, lib=lib)
    assert z == 0.0 and math.copysign(1.0, z) < 0
    assert oracle.half_to_double(0x7C00, lib=lib) == math.inf
    assert oracle.half_to_double(0xFC00, lib=lib) == -math.inf
    assert math.isnan(oracle.half_to_double(0x7E00, lib=lib))


def check_half_all_patterns(lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    # decode through the oracle's gather: a [65536,1,1,1] pool, one head
    pool = bits.reshape(-1, 1, 1, 1)
    got = oracle.gather(pool, np.arange(1 << 16, dtype=np.int32), 1 << 16, 0, lib=lib)[:, 0]
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def _replay_case(case, lib):
    nb, bs, hd = case["num_blocks"], case["block_size"], case["head_dim"]
    alloc = BlockAllocator(nb, bs)
    seq = Sequence_(0, case["prompt_len"])
    if "expect_error" in case:
        with pytest.raises(RuntimeError) as ei:
            alloc.allocate_for_prefill(seq)
        assert case["expect_error"] in str(ei.value)
        assert seq.block_table == [] and len(alloc.free_blocks) == nb
        return
    alloc.allocate_for_prefill(seq)
    ap = case["after_prefill"]
    assert len(seq.block_table) == ap["table_len"]
    if "free" in ap:
        assert len(alloc.free_blocks) == ap["free"]
    done = 0
    for chk in case["decode_checks"]:
        while done < chk["decodes"]:
            alloc.allocate_for_decode(seq)
            done += 1
        assert seq.seq_len == chk["seq_len"]
        assert len(seq.block_table) == chk["table_len"]
        if "free" in chk:
            assert len(alloc.free_blocks) == chk["free"]
    # the notes' single-head pool [num_blocks, block_size, head_dim] = H=1
    pool = np.zeros((nb, bs, 1, hd), np.float16)
    for blk, val in zip(seq.block_table, case["fill_values"]):
        pool[blk] = val
    got = oracle.gather(pool, np.asarray(seq.block_table, np.int32), seq.seq_len, 0, lib=lib)
    assert list(got.shape) == case["gathered_shape"]
    for lo, hi, val in case["gathered_ranges"]:
        assert np.all(got[lo:hi] == val)
    return seq, pool, alloc


def check_worked_examples(lib):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        _replay_case(case, lib)


def check_closed_form_uniform(lib):
    """q = 0: all scores equal, output = mean of visible V rows.  With the
    notes' fill patterns: (4*1 + 4*2 + 1*3)/9 and (4*7 + 1*8)/5."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    expect = {"prefill_decode_gather": 15.0 / 9.0, "block_boundary": 36.0 / 5.0}
    for case in cases:
        if case["name"] not in expect:
            continue
        seq, vpool, _ = _replay_case(case, lib)
        hd = case["head_dim"]
        kpool = rand16(np.random.default_rng(5), vpool.shape)
        q = np.zeros((1, 1, hd), np.float16)
        out = oracle.decode(q, kpool, vpool, np.asarray([seq.block_table], np.int32),
                            [seq.seq_len], 1.0 / math.sqrt(hd), lib=lib)
        assert np.allclose(out, expect[case["name"]], rtol=0, atol=1e-14)


def check_single_key_and_ones(lib):
    rng = np.random.default_rng(11)
    k, v, tables, _ = paged_case(rng, 2, 3, 64, 4, [1, 13])
    q = rand16(rng, (2, 3, 64))
    out = oracle.decode(q, k, v, tables, [1, 13], 0.125, lib=lib)
    # one key -> exactly that key's value row
    assert np.array_equal(out[0], v[tables[0, 0], 0].astype(np.float64))
    # V = 1 -> rows of 1 (weights sum to one)
    ones = np.ones_like(v)
    out1 = oracle.decode(q, k, ones, tables, [1, 13], 0.125, lib=lib)
    assert np.allclose(out1, 1.0, rtol=0, atol=1e-14)


def check_two_keys_logistic(lib):
    rng = np.random.default_rng(12)
    D = 8
    k, v, tables, _ = paged_case(rng, 1, 1, D, 4, [2], spare=0)
    q = rand16(rng, (1, 1, D))
    scale = 0.3
    k0 = k[tables[0, 0], 0, 0].astype(np.float64)
    k1 = k[tables[0, 0], 1, 0].astype(np.float64)
    qq = q[0, 0].astype(np.float64)
    s0 = scale * sum(float(a) * float(b) for a, b in zip(qq, k0))
    s1 = scale * sum(float(a) * float(b) for a, b in zip(qq, k1))
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expect = w0 * v[tables[0, 0], 0, 0].astype(np.float64) + w1 * v[tables[0, 0], 1, 0].astype(np.float64)
    out = oracle.decode(q, k, v, tables, [2], scale, lib=lib)
    assert np.allclose(out[0, 0], expect, rtol=1e-13, atol=1e-14)


def check_scale_zero_mean(lib):
    rng = np.random.default_rng(13)
    k, v, tables, ctx = paged_case(rng, 3, 2, 16, 4, [5, 1, 11])
    q = rand16(rng, (3, 2, 16))
    out = oracle.decode(q, k, v, tables, ctx, 0.0, lib=lib)
    for b in range(3):
        for h in range(2):
            mean = contiguous(v, tables[b], ctx[b], h).mean(axis=0)
            assert np.allclose(out[b, h], mean, rtol=1e-13, atol=1e-14)


def check_dense_decode(lib):
    rng = np.random.default_rng(14)
    for (B, H, D, bs, ctx) in [(3, 2, 16, 4, [5, 9, 1]), (2, 3, 32, 16, [17, 40]),
                               (4, 1, 8, 32, [33, 64, 2, 31])]:
        k, v, tables, ctx = paged_case(rng, B, H, D, bs, ctx)
        q = rand16(rng, (B, H, D))
        scale = 1.0 / math.sqrt(D) * 1.7
        out = oracle.decode(q, k, v, tables, ctx, scale, lib=lib)
        for b in range(B):
            for h in range(H):
                K = contiguous(k, tables[b], ctx[b], h)
                V = contiguous(v, tables[b], ctx[b], h)
                ref = dense_attention(q[b, h][None].astype(np.float64), K, V, scale)[0]
                assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)


def check_dense_prefill(lib):
    rng = np.random.default_rng(15)
    for (B, H, D, bs, Lq, ctx) in [(2, 2, 16, 4, 3, [7, 3]), (1, 2, 32, 16, 20, [45]),
                                   (2, 1, 8, 4, 1, [9, 4])]:
        k, v, tables, ctx = paged_case(rng, B, H, D, bs, ctx)
        q = rand16(rng, (B, H, Lq, D))
        scale = 0.2
        out = oracle.prefill(q, k, v, tables, ctx, scale, lib=lib)
        for b in range(B):
            n = int(ctx[b])
            # query i of the chunk sits at position n-Lq+i and sees keys <= it
            mask = np.arange(n)[None, :] <= (n - Lq + np.arange(Lq))[:, None]
            for h in range(H):
                K = contiguous(k, tables[b], n, h)
                V = contiguous(v, tables[b], n, h)
                ref = dense_attention(q[b, h].astype(np.float64), K, V, scale, mask)
                assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)


def check_prefill_whole_context_is_tril(lib):
    """Lq == ctx: the lower-triangular mask of the blog's sec. 3.2.2."""
    rng = np.random.default_rng(16)
    k, v, tables, ctx = paged_case(rng, 1, 1, 8, 4, [6])
    q = rand16(rng, (1, 1, 6, 8))
    out = oracle.prefill(q, k, v, tables, ctx, 0.5, lib=lib)
    tril = np.tril(np.ones((6, 6), bool))
    K = contiguous(k, tables[0], 6, 0)
    V = contiguous(v, tables[0], 6, 0)
    ref = dense_attention(q[0, 0].astype(np.float64), K, V, 0.5, tril)
    assert np.allclose(out[0, 0], ref, rtol=1e-12, atol=1e-13)
    # row 0 sees only key 0
    assert np.array_equal(out[0, 0, 0], V[0])


def check_prefill_lq1_is_decode(lib):
    rng = np.random.default_rng(17)
    k, v, tables, ctx = paged_case(rng, 3, 2, 16, 4, [5, 9, 1])
    q = rand16(rng, (3, 2, 1, 16))
    a = oracle.prefill(q, k, v, tables, ctx, 0.25, lib=lib)[:, :, 0]
    b = oracle.decode(q[:, :, 0], k, v, tables, ctx, 0.25, lib=lib)
    assert np.array_equal(a, b)


def check_prefill_varlen_rows_are_decodes(lib):
    """Query i of a chunk of n new queries on a context of c keys is a decode
    over keys 0 .. c-n+i; padded rows are zero; equal lengths give prefill."""
    rng = np.random.default_rng(27)
    B, H, D, bs, Lq = 4, 2, 16, 4, 6
    k, v, tables, ctx = paged_case(rng, B, H, D, bs, [9, 6, 13, 3])
    q = rand16(rng, (B, H, Lq, D))
    q_lens = [4, 6, 0, 3]
    out = oracle.prefill_varlen(q, k, v, tables, ctx, q_lens, 0.3, lib=lib)
    for b in range(B):
        n, c = q_lens[b], int(ctx[b])
        assert np.all(out[b, :, n:] == 0.0)
        for i in range(n):
            row = oracle.decode(q[b:b + 1, :, i], k, v, tables[b:b + 1], [c - n + i + 1], 0.3,
                                lib=lib)[0]
            assert np.array_equal(out[b, :, i], row)
    full = oracle.prefill_varlen(q[:, :, :3], k, v, tables, ctx, [3, 3, 3, 3], 0.3, lib=lib)
    assert np.array_equal(full, oracle.prefill(q[:, :, :3], k, v, tables, ctx, 0.3, lib=lib))
    with pytest.raises(oracle.OracleError):  # more new queries than keys
        oracle.prefill_varlen(q, k, v, tables, ctx, [4, 6, 0, 4], 0.3, lib=lib)


def check_permutation_invariance(lib):
    rng = np.random.default_rng(18)
    k, v, tables, ctx = paged_case(rng, 3, 2, 16, 4, [7, 12, 3], spare=5)
    q = rand16(rng, (3, 2, 16))
    out = oracle.decode(q, k, v, tables, ctx, 0.25, lib=lib)
    perm = rng.permutation(k.shape[0])           # old id -> new id
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = oracle.decode(q, k2, v2, t2, ctx, 0.25, lib=lib)
    assert np.array_equal(out, out2)


def check_cache_write(lib):
    rng = np.random.default_rng(19)
    nb, bs, H, D = 6, 4, 2, 8
    kc = rand16(rng, (nb, bs, H, D))
    vc = rand16(rng, (nb, bs, H, D))
    slots = np.array([5, 0, -1, 23, 9], np.int64)
    kn = rand16(rng, (5, H, D))
    vn = rand16(rng, (5, H, D))
    k2, v2 = oracle.kv_cache_write(kn, vn, slots, kc, vc, lib=lib)
    ek = kc.view(np.uint16).copy().reshape(nb * bs, H, D)
    ev = vc.view(np.uint16).copy().reshape(nb * bs, H, D)
    for t, s in enumerate(slots):
        if s >= 0:
            ek[s] = kn[t].view(np.uint16)
            ev[s] = vn[t].view(np.uint16)
    assert np.array_equal(k2.reshape(nb * bs, H, D), ek)
    assert np.array_equal(v2.reshape(nb * bs, H, D), ev)


def check_block_copy(lib):
    rng = np.random.default_rng(20)
    nb, bs, H, D = 8, 4, 2, 8
    kc = rand16(rng, (nb, bs, H, D))
    vc = rand16(rng, (nb, bs, H, D))
    pairs = np.array([[1, 4], [1, 5], [6, 6], [2, 0]], np.int64)
    k2, v2 = oracle.block_copy(kc, vc, pairs, lib=lib)
    ek, ev = kc.view(np.uint16).copy(), vc.view(np.uint16).copy()
    for s, d in pairs:
        ek[d] = kc.view(np.uint16)[s]
        ev[d] = vc.view(np.uint16)[s]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


# ---- FP8 (e4m3) storage -------------------------------------------------------
E4M3_KNOWN = {0x00: 0.0, 0x38: 1.0, 0x30: 0.5, 0x7E: 448.0, 0x01: 2.0 ** -9,
              0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x39: 1.125, 0x3F: 1.875,
              0xB8: -1.0, 0xFE: -448.0, 0x40: 2.0}


def check_e4m3_decode(lib):
    for code, val in E4M3_KNOWN.items():
        assert oracle.e4m3_to_double(code, lib=lib) == val, hex(code)
    assert math.isnan(oracle.e4m3_to_double(0x7F, lib=lib))
    assert math.isnan(oracle.e4m3_to_double(0xFF, lib=lib))
    import torch
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c, lib=lib) for c in range(256)])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin]) and np.array_equal(np.isnan(got), np.isnan(ref))


def check_e4m3_encode(lib):
    # every finite code round-trips
    for c in range(256):
        v = oracle.e4m3_to_double(c, lib=lib)
        if math.isfinite(v):
            got = oracle.e4m3_from_float(v, lib=lib)
            assert got == c or (v == 0.0 and got in (0x00, 0x80)), (hex(c), hex(got))
    # ties go to the even code; just past a tie goes up; saturation at 448
    assert oracle.e4m3_from_float(1.0625, lib=lib) == 0x38
    assert oracle.e4m3_from_float(1.1875, lib=lib) == 0x3A
    assert oracle.e4m3_from_float(np.nextafter(np.float32(1.0625), np.float32(2)), lib=lib) == 0x39
    assert oracle.e4m3_from_float(1000.0, lib=lib) == 0x7E
    assert oracle.e4m3_from_float(-1000.0, lib=lib) == 0xFE
    # torch's float32 -> float8_e4m3fn (round to nearest even) on in-range values
    import torch
    x = np.random.default_rng(30).standard_normal(2000).astype(np.float32) * 50
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(v, lib=lib) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def _fp8_case(rng, nb=6, bs=4, H=2, D=16):
    k8 = np.zeros((nb, bs, H, D), np.uint8)
    v8 = np.zeros_like(k8)
    ks = np.ones((nb, H, bs), np.float32)
    vs = np.ones_like(ks)
    return k8, v8, ks, vs


def check_fp8_quantize(lib):
    rng = np.random.default_rng(31)
    k8, v8, ks, vs = _fp8_case(rng)
    T, H, D = 5, 2, 16
    k = rand16(rng, (T, H, D)) * np.float16(3)
    v = rand16(rng, (T, H, D))
    v[2, 1] = 0  # an all-zero row: scale 1, codes 0
    slots = np.array([0, 5, 9, 23, -1], np.int64)
    k8, v8, ks, vs = oracle.kv_cache_write_fp8(k, v, slots, k8, v8, ks, vs, lib=lib)
    bs = 4
    for t, sl in enumerate(slots[:4]):
        blk, off = sl // bs, sl % bs
        for h in range(H):
            for x, codes, sc in ((k[t, h], k8[blk, off, h], ks[blk, h, off]),
                                 (v[t, h], v8[blk, off, h], vs[blk, h, off])):
                xf = x.astype(np.float32)
                amax = np.float32(np.abs(xf).max())
                assert sc == (amax / np.float32(448) if amax > 0 else 1.0)
                dec = np.array([oracle.e4m3_to_double(c, lib=lib) for c in codes])
                deq = dec * sc
                if amax > 0:  # the max element maps to +-448; 448 * scale ~ max within 1 ulp
                    assert np.max(np.abs(dec)) == 448.0
                    assert abs(np.max(np.abs(deq)) - float(amax)) <= float(amax) * 2.0 ** -23
                err = np.abs(deq - xf.astype(np.float64))
                assert np.all(err <= np.abs(xf) * 2.0 ** -4 + 2.0 ** -10 * sc)
    assert np.all(v8[9 // bs, 9 % bs, 1] == 0) and vs[9 // bs, 1, 9 % bs] == 1.0


def check_fp8_decode_dense(lib):
    rng = np.random.default_rng(32)
    B, H, D, bs = 3, 2, 16, 4
    ctx = [5, 9, 1]
    nb = 8
    k8 = rng.integers(0, 0x7E, size=(nb, bs, H, D), dtype=np.uint8) | \
        (rng.integers(0, 2, size=(nb, bs, H, D), dtype=np.uint8) << 7)
    v8 = rng.integers(0, 0x7E, size=(nb, bs, H, D), dtype=np.uint8)
    ks = (rng.random((nb, H, bs)) * 0.01 + 0.001).astype(np.float32)
    vs = (rng.random((nb, H, bs)) * 0.01 + 0.001).astype(np.float32)
    perm = rng.permutation(nb)
    tables = np.full((B, 3), -1, np.int32)
    pos = 0
    for b, c in enumerate(ctx):
        n = -(-c // bs)
        tables[b, :n] = perm[pos:pos + n]
        pos += n
    q = rand16(rng, (B, H, D))
    out = oracle.decode_fp8(q, k8, v8, ks, vs, tables, ctx, 0.3, lib=lib)
    dec = np.vectorize(lambda c: oracle.e4m3_to_double(int(c), lib=lib))
    for b in range(B):
        j = np.arange(ctx[b])
        blk, off = tables[b, j // bs], j % bs
        for h in range(H):
            K = dec(k8[blk, off, h, :]) * ks[blk, h, off][:, None]
            V = dec(v8[blk, off, h, :]) * vs[blk, h, off][:, None]
            ref = dense_attention(q[b, h][None].astype(np.float64), K, V, 0.3)[0]
            assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-14)


ALL_CHECKS = [
    check_half_known, check_half_all_patterns, check_worked_examples,
    check_closed_form_uniform, check_single_key_and_ones,
    check_two_keys_logistic, check_scale_zero_mean, check_dense_decode,
    check_dense_prefill, check_prefill_whole_context_is_tril,
    check_prefill_lq1_is_decode, check_prefill_varlen_rows_are_decodes,
    check_permutation_invariance,
    check_cache_write, check_block_copy, check_e4m3_decode, check_e4m3_encode,
    check_fp8_quantize, check_fp8_decode_dense,
]


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check, lib):
    check(lib)


# ----------------------------------------------------------------------------
# error behaviour
# ----------------------------------------------------------------------------
def test_oracle_rejects_bad_inputs(lib):
    rng = np.random.default_rng(21)
    k, v, tables, ctx = paged_case(rng, 2, 1, 8, 4, [5, 3])
    q = rand16(rng, (2, 1, 8))
    bad = tables.copy()
    bad[0, 1] = k.shape[0]  # out of range, needed for ctx 5
    with pytest.raises(oracle.OracleError) as ei:
        oracle.decode(q, k, v, bad, ctx, 1.0, lib=lib)
    assert ei.value.code == 2
    # entries past ceil(ctx / bs) are never read, even if garbage
    junk = tables.copy()
    junk[1, 1:] = 123456
    oracle.decode(q, k, v, junk, ctx, 1.0, lib=lib)
    with pytest.raises(oracle.OracleError):
        oracle.decode(q, k, v, tables, [-1, 3], 1.0, lib=lib)
    with pytest.raises(oracle.OracleError):  # more keys than the table holds
        oracle.decode(q, k, v, tables, [5, 3 + 4 * tables.shape[1]], 1.0, lib=lib)
    # ctx == 0 -> zero row
    out = oracle.decode(q, k, v, tables, [0, 3], 1.0, lib=lib)
    assert np.all(out[0] == 0.0)
    kn = rand16(rng, (2, 1, 8))
    with pytest.raises(oracle.OracleError) as ei:
        oracle.kv_cache_write(kn, kn, np.array([3, 3]), k, v, lib=lib)
    assert ei.value.code == 5
    with pytest.raises(oracle.OracleError) as ei:
        oracle.kv_cache_write(kn, kn, np.array([3, k.shape[0] * 4]), k, v, lib=lib)
    assert ei.value.code == 4
    for pairs in ([[0, 1], [2, 1]], [[0, 1], [1, 2]], [[0, k.shape[0]]]):
        with pytest.raises(oracle.OracleError) as ei:
            oracle.block_copy(k, v, np.array(pairs), lib=lib)
        assert ei.value.code == 6


# ----------------------------------------------------------------------------
# allocator behaviour beyond the worked examples
# ----------------------------------------------------------------------------
def test_allocator_waste_and_free():
    bs = 16
    rng = np.random.default_rng(22)
    alloc = BlockAllocator(400, bs, rng.permutation(400))
    seqs = []
    for i, n in enumerate(rng.integers(1, 300, size=12)):
        s = Sequence_(i, int(n))
        alloc.allocate_for_prefill(s)
        for _ in range(int(rng.integers(0, 40))):
            alloc.allocate_for_decode(s)
        assert 0 <= alloc.wasted_slots(s) <= bs - 1
        seqs.append(s)
    used = sum(len(s.block_table) for s in seqs)
    assert alloc.in_use() == used and len(alloc.free_blocks) == 400 - used
    ids = [b for s in seqs for b in s.block_table]
    assert len(set(ids)) == len(ids)
    for s in seqs:
        alloc.free(s)
    assert len(alloc.free_blocks) == 400 and alloc.in_use() == 0


def test_allocator_oom_is_atomic():
    alloc = BlockAllocator(3, 4)
    a = Sequence_(0, 8)
    alloc.allocate_for_prefill(a)
    b = Sequence_(1, 9)
    with pytest.raises(OutOfBlocks, match="OOM"):
        alloc.allocate_for_prefill(b)
    assert b.block_table == [] and len(alloc.free_blocks) == 1
    c = Sequence_(2, 4)
    alloc.allocate_for_prefill(c)
    with pytest.raises(OutOfBlocks, match="OOM"):
        alloc.allocate_for_decode(c)
    assert c.seq_len == 4 and len(c.block_table) == 1


def test_allocator_bs1_growth_reading():
    alloc = BlockAllocator(5, 1)
    s = Sequence_(0, 2)
    alloc.allocate_for_prefill(s)
    alloc.allocate_for_decode(s)
    assert len(s.block_table) == 3 == s.seq_len


def test_allocator_fork_cow():
    alloc = BlockAllocator(12, 4)
    parent = Sequence_(0, 8)
    alloc.allocate_for_prefill(parent)
    kids = [alloc.fork(parent, i + 1) for i in range(3)]
    assert all(k.block_table == parent.block_table for k in kids)
    assert alloc.refcount[parent.block_table[1]] == 4
    pairs = [alloc.copy_on_write(k, 1) for k in kids]
    assert all(p is not None and p[0] == parent.block_table[1] for p in pairs)
    assert len({p[1] for p in pairs}) == 3
    assert alloc.refcount[parent.block_table[1]] == 1
    assert alloc.copy_on_write(parent, 1) is None
    for k in kids:
        alloc.free(k)
    alloc.free(parent)
    assert len(alloc.free_blocks) == 12


# ----------------------------------------------------------------------------
# mutation tests: each planted mistake must fail at least one pin
# ----------------------------------------------------------------------------
MUTANTS = {
    "drop_scale": ("pool_at(k_cache, blk, tok, head, d, bs, H, D);\n        s[j] = scale * dot;",
                   "pool_at(k_cache, blk, tok, head, d, bs, H, D);\n        s[j] = dot;"),
    "token_index_swapped": ("int tok = j % bs;\n        double dot", "int tok = j / bs;\n        double dot"),
    "no_normalisation": ("double w = s[j] / z;\n        for (int d = 0; d < D; ++d)\n            out[d]",
                         "double w = s[j];\n        for (int d = 0; d < D; ++d)\n            out[d]"),
    "mask_off_by_one": ("ctx - Lq + i + 1", "ctx - Lq + i"),
    "head_row_swapped": ("(((blk * bs + tok) * (int64_t)H + head) * D) + d",
                         "(((blk * bs + head) * (int64_t)H + tok) * D) + d"),
    "exponent_bias": ("ldexp((double)(1024 + frac), e - 25)", "ldexp((double)(1024 + frac), e - 24)"),
    "subnormal_scale": ("ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    "max_not_subtracted_wrong_sign": ("        s[j] = exp(s[j] - m);\n        z += s[j];\n    }\n    /* weighted",
                                      "        s[j] = exp(m - s[j]);\n        z += s[j];\n    }\n    /* weighted"),
    "fp8_no_normalisation": ("double w = s[j] / z;\n                for",
                             "double w = s[j];\n                for"),
    "write_wrong_pool": ("v_cache[slot * row + e] = v[(int64_t)t * row + e];",
                         "v_cache[slot * row + e] = k[(int64_t)t * row + e];"),
    "copy_reversed": ("memcpy(k_cache + dst * blk, k_cache + src * blk",
                      "memcpy(k_cache + src * blk, k_cache + dst * blk"),
    "e4m3_bias": ("ldexp((double)(8 + frac), e - 10)", "ldexp((double)(8 + frac), e - 11)"),
    "e4m3_tie_up": ("pick = (lo & 1) ? hi : lo;", "pick = hi;"),
    "fp8_scale_index": ("double kscale = (double)ks[(blk * H + h) * bs + off];",
                        "double kscale = (double)ks[(blk * bs + off) * H + h];"),
    "fp8_scale_max": ("float s = amax > 0.0f ? amax / 448.0f : 1.0f;",
                      "float s = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    "first_key_skipped": ("for (int j = 0; j < n_keys; ++j) {\n        int64_t blk = table[j / bs];\n        int tok = j % bs;\n        double w",
                          "for (int j = 1; j < n_keys; ++j) {\n        int64_t blk = table[j / bs];\n        int tok = j % bs;\n        double w"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    with open(obuild.SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutant = oracle.load(obuild.build_variant(src.replace(old, new), f"mutant_{name}"))
    failed = []
    for check in ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, oracle.OracleError, pytest.fail.Exception):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
