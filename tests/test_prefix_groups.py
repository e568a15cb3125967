"""pa_shared_prefix_groups (host code): groups derived from the block tables
are valid CSR groups whose shared lengths are the members' exact longest
common prefixes, checked against brute force over the tables; without a
group-size cap they are exactly the classes of sequences agreeing on their
first ceil(min_shared_tokens / block_size) blocks."""
import numpy as np
import pytest
import torch

import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import build_lib, workloads


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    return pk.lib()


def chains(tables, ctx, bs):
    """Each sequence's full blocks (stopping at the first -1)."""
    out = []
    cap = tables.shape[1] * bs
    for row, n in zip(tables, ctx):
        full = max(0, min(int(n), cap)) // bs
        c = []
        for x in row[:full]:
            if x < 0:
                break
            c.append(int(x))
        out.append(tuple(c))
    return out


def lcp(a, b):
    n = 0
    while n < min(len(a), len(b)) and a[n] == b[n]:
        n += 1
    return n


def groups_of(tables, ctx, bs, min_tokens=0, gmax=16):
    sg, off, seqs, plen = pk.pa_shared_prefix_groups(torch.from_numpy(tables),
                                                     torch.from_numpy(ctx), bs, min_tokens,
                                                     gmax)
    G = plen.numel()
    members = [seqs[off[g]:off[g + 1]].tolist() for g in range(G)]
    return sg.tolist(), members, plen.tolist()


def check_valid(tables, ctx, bs, min_tokens, gmax):
    sg, members, plen = groups_of(tables, ctx, bs, min_tokens, gmax)
    ch = chains(tables, ctx, bs)
    seen = set()
    min_blocks = max(1, -(-min_tokens // bs))
    for g, m in enumerate(members):
        assert 2 <= len(m) <= gmax
        assert m == sorted(m)
        assert not seen & set(m)
        seen |= set(m)
        for s in m:
            assert sg[s] == g
        shared = min(lcp(ch[m[0]], ch[s]) for s in m[1:])
        # the shared length is the exact longest common prefix of the members
        assert plen[g] == shared * bs
        assert shared >= min_blocks
        # every member's context holds the prefix
        assert all(int(ctx[s]) >= plen[g] for s in m)
    assert all(sg[s] == -1 for s in range(len(ctx)) if s not in seen)
    return sg, members, plen


def test_prefix_sharing_layout_gives_its_groups():
    lay = workloads.prefix_sharing_layout(seed=2)
    want = workloads.sharing_groups(lay)
    got = pk.pa_shared_prefix_groups(torch.from_numpy(lay.tables),
                                     torch.from_numpy(lay.context_lens), lay.block_size, 0, 16)
    for w, g in zip(want, got):
        assert np.array_equal(w, g.numpy())


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("min_blocks", [1, 3])
def test_uncapped_groups_are_classes_of_the_first_blocks(seed, min_blocks):
    bs = 16
    tables, ctx, _ = workloads.fork_forest_layout(seed, B=40, block_size=bs)
    sg, members, plen = check_valid(tables, ctx, bs, min_blocks * bs - 5, gmax=1000)
    ch = chains(tables, ctx, bs)
    classes = {}
    for s, c in enumerate(ch):
        if len(c) >= min_blocks:
            classes.setdefault(c[:min_blocks], []).append(s)
    want = sorted(m for m in classes.values() if len(m) >= 2)
    assert sorted(members) == want


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("gmax", [2, 3, 5, 64])
def test_capped_groups_are_valid(seed, gmax):
    bs = 32
    tables, ctx, _ = workloads.fork_forest_layout(100 + seed, B=60, block_size=bs, p_root=0.05)
    first = check_valid(tables, ctx, bs, 0, gmax)
    assert groups_of(tables, ctx, bs, 0, gmax) == first  # deterministic
    # every sequence sharing its first block with another is grouped when the
    # cap does not bind
    if gmax >= len(ctx):
        ch = chains(tables, ctx, bs)
        firsts = [c[:1] for c in ch]
        for s, f in enumerate(firsts):
            if f and firsts.count(f) >= 2:
                assert first[0][s] >= 0


def test_oversized_node_prefers_deeper_subgroups():
    # 20 sequences share blocks 0..3; sequences 0..2 share 0..5; cap 16:
    # {0,1,2} at 6 blocks, then 3..18 at 4 blocks; 19 is left over alone
    bs = 16
    B = 20
    tables = np.full((B, 8), -1, np.int32)
    nxt = 100
    for b in range(B):
        tables[b, :4] = [7, 3, 9, 1]
        if b < 3:
            tables[b, 4:6] = [40, 41]
            tables[b, 6] = nxt
            nxt += 1
        else:
            tables[b, 4] = nxt
            nxt += 1
    ctx = np.array([7 * bs if b < 3 else 5 * bs for b in range(B)], np.int32)
    sg, members, plen = check_valid(tables, ctx, bs, 0, 16)
    assert members == [[0, 1, 2], list(range(3, 19))]
    assert plen == [6 * bs, 4 * bs]
    assert sg[19] == -1


def test_partial_last_block_and_sentinel_are_not_shared():
    bs = 16
    tables = np.array([[5, 6, 7, -1],
                       [5, 6, 7, -1],
                       [5, 6, -1, 7],
                       [8, 9, 10, 11]], np.int32)
    # seq 0: 2 full blocks + part of block 7; seq 1: 3 full; seq 2 stops at -1
    ctx = np.array([2 * bs + 3, 3 * bs, 4 * bs, 4 * bs], np.int32)
    sg, members, plen = check_valid(tables, ctx, bs, 0, 16)
    assert members == [[0, 1, 2]] and plen == [2 * bs]
    # a context longer than the table caps at the table: seqs 0 and 1 now
    # share three full blocks, but seq 2 leaves them after two, so the three
    # form one group at the node where they part
    ctx2 = np.array([100 * bs] * 4, np.int32)
    assert groups_of(tables, ctx2, bs)[1:] == ([[0, 1, 2]], [2 * bs])
    # with a minimum of three blocks only the pair remains
    assert groups_of(tables, ctx2, bs, 3 * bs)[1:] == ([[0, 1]], [3 * bs])


def test_min_shared_tokens_filters_short_prefixes():
    bs = 16
    tables = np.array([[1, 2, 3, 4], [1, 2, 3, 5], [1, 9, 10, 11], [6, 7, 8, 12]], np.int32)
    ctx = np.full(4, 4 * bs, np.int32)
    assert groups_of(tables, ctx, bs, 0)[1] == [[0, 1, 2]]
    assert groups_of(tables, ctx, bs, 2 * bs)[1:] == ([[0, 1]], [3 * bs])
    assert groups_of(tables, ctx, bs, 3 * bs + 1)[1] == []


def test_degenerate_inputs():
    bs = 16
    e = np.zeros((0, 4), np.int32)
    sg, off, seqs, plen = pk.pa_shared_prefix_groups(torch.from_numpy(e),
                                                     torch.zeros(0, dtype=torch.int32), bs)
    assert sg.numel() == 0 and off.tolist() == [0] and seqs.numel() == 0 and plen.numel() == 0
    one = np.array([[1, 2]], np.int32)
    assert groups_of(one, np.array([32], np.int32), bs)[1] == []
    # zero and negative lengths hold no blocks
    two = np.array([[1, 2], [1, 2]], np.int32)
    assert groups_of(two, np.array([0, -5], np.int32), bs)[1] == []
    assert groups_of(two, np.array([16, 40], np.int32), bs)[1:] == ([[0, 1]], [16])


def test_invalid_arguments_return_invalid(_lib):
    import ctypes
    G = ctypes.c_int(7)
    buf = (ctypes.c_int32 * 16)()
    ok = dict(bt=buf, cl=buf, B=2, M=2, bs=16, mn=0, gm=16)

    def rc(**kw):
        a = dict(ok, **kw)
        return _lib.pa_shared_prefix_groups(a["bt"], a["cl"], a["B"], a["M"], a["bs"], a["mn"],
                                            a["gm"], buf, buf, buf, buf, ctypes.byref(G))
    for kw in (dict(B=-1), dict(M=0), dict(bs=0), dict(mn=-1), dict(gm=1), dict(bt=None)):
        G.value = 7
        assert rc(**kw) == pk.PA_ERR_INVALID, kw
        assert G.value == 0
    assert _lib.pa_shared_prefix_groups(buf, buf, 2, 2, 16, 0, 16, buf, buf, buf, buf,
                                        None) == pk.PA_ERR_INVALID
