"""fp64 CPU oracle for paged attention and the paged-cache copy operations.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It never imports
or calls the CUDA library, and the CUDA library never calls it.

The arithmetic lives in ``pa_oracle.c`` (plain C, IEEE binary64, left to
right summation); this module only marshals numpy arrays into it.  fp16
inputs are passed as their raw 16-bit patterns and decoded exactly in C.

Functions and the passages they follow (page titles and sections):
  attend_row / decode / prefill / prefill_varlen -- blog "PagedAttention origin and evolution"
      sec. 3.2.2 (forward pass: gather through the block table, scale by
      1/sqrt(head_dim), softmax, weighted V) and tutorial chapter
      "4. PagedAttention机制：vLLM的核心创新", section "PagedAttention的注意力计算";
      prefill uses the end-aligned causal reading of the sec. 3.2.2 mask;
      prefill_varlen is that prefill per sequence on its own chunk length
      (the sec. 3.2.2 forward pass takes each request's queries separately).
  kv_cache_write -- the same tutorial, section "Block管理策略" (the cache grows
      into newly mapped blocks); slot = physical_block * block_size + offset.
  block_copy -- study notes "DataWhale组队学习笔记--llm-algo-leetcode(五)",
      "4. PagedAttention 带来的核心红利" (copy-on-write of shared blocks).
  gather -- the same notes, "代码实现" (get_physical_cache).
  e4m3_* / kv_cache_write_fp8 / decode_fp8 -- the blog's sec. 2.3 "mixed
      precision KV storage", read as e4m3 codes with one fp32 scale per
      (token, head) row (scale = max|row| / 448); decode dequantizes exactly.
  allocator.BlockAllocator -- the same notes' KVCacheManager plus the
      tutorial's Free List / Allocator table.
"""
import ctypes

import numpy as np

from . import build as _build

__all__ = [
    "OracleError", "half_to_double", "attend_row", "decode", "prefill", "prefill_varlen",
    "kv_cache_write", "block_copy", "gather", "load", "e4m3_to_double", "e4m3_from_float",
    "kv_cache_write_fp8", "decode_fp8",
]

_ERRORS = {
    1: "bad argument",
    2: "block-table entry out of range",
    3: "bad context length",
    4: "slot out of range",
    5: "duplicate slot",
    6: "bad or overlapping copy pair",
}


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle error {code}: {_ERRORS.get(code, '?')}")
        self.code = code


_lib = None
_P = ctypes.c_void_p


def _bind(lib):
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_attend_row.argtypes = [_P, _P, _P, _P, i32, i32, i32, i32, i32,
                                      i32, i64, dbl, _P]
    lib.oracle_decode.argtypes = [_P, _P, _P, _P, _P, i32, i32, i32, i32, i64,
                                  i32, dbl, _P]
    lib.oracle_prefill.argtypes = [_P, _P, _P, _P, _P, i32, i32, i32, i32,
                                   i32, i64, i32, dbl, _P]
    lib.oracle_kv_cache_write.argtypes = [_P, _P, _P, i32, i32, i32, i32, i64,
                                          _P, _P]
    lib.oracle_block_copy.argtypes = [_P, _P, _P, i32, i32, i32, i32, i64]
    lib.oracle_gather.argtypes = [_P, _P, i32, i32, i32, i32, i32, i32, i64, _P]
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
    lib.oracle_kv_cache_write_fp8.argtypes = [_P, _P, _P, i32, i32, i32, i32, i64, _P, _P, _P, _P]
    lib.oracle_decode_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, i32, i32, i32, i32, i64, i32,
                                      dbl, _P]
    for f in ("oracle_attend_row", "oracle_decode", "oracle_prefill",
              "oracle_kv_cache_write", "oracle_block_copy", "oracle_gather",
              "oracle_kv_cache_write_fp8", "oracle_decode_fp8"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def load(path=None):
    """Load (building first if needed) the oracle library.  ``path`` loads a
    specific build, e.g. a test's deliberately broken copy."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bits(a):
    """fp16 array -> contiguous uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 or uint16 bits, got {a.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc != 0:
        raise OracleError(rc)


def half_to_double(bits, lib=None):
    lib = lib or load()
    return lib.oracle_half_to_double(int(bits) & 0xFFFF)


def attend_row(q_row, k_cache, v_cache, table, n_keys, head, scale, lib=None):
    """One query row of one head attending to logical keys 0..n_keys-1.
    k_cache/v_cache: [num_blocks, block_size, H, D] fp16; table: int32."""
    lib = lib or load()
    kc, vc = _bits(k_cache), _bits(v_cache)
    nb, bs, H, D = kc.shape
    q = _bits(q_row).reshape(D)
    tb = np.ascontiguousarray(table, dtype=np.int32)
    out = np.zeros(D, dtype=np.float64)
    _check(lib.oracle_attend_row(_ptr(q), _ptr(kc), _ptr(vc), _ptr(tb),
                                 int(tb.size), int(n_keys), H, int(head), D,
                                 bs, nb, float(scale), _ptr(out)))
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, lib=None):
    """q[B,H,D] fp16 -> out[B,H,D] fp64."""
    lib = lib or load()
    qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    B, H, D = qb.shape
    nb, bs = kc.shape[0], kc.shape[1]
    assert kc.shape == (nb, bs, H, D) and vc.shape == kc.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(B, -1)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32).reshape(B)
    out = np.zeros((B, H, D), dtype=np.float64)
    _check(lib.oracle_decode(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                             B, H, D, bs, nb, bt.shape[1], float(scale),
                             _ptr(out)))
    return out


def prefill(q, k_cache, v_cache, block_tables, context_lens, scale, lib=None):
    """q[B,H,Lq,D] fp16 (the last Lq positions of each context) ->
    out[B,H,Lq,D] fp64 with the end-aligned causal mask."""
    lib = lib or load()
    qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    B, H, Lq, D = qb.shape
    nb, bs = kc.shape[0], kc.shape[1]
    assert kc.shape == (nb, bs, H, D) and vc.shape == kc.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(B, -1)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32).reshape(B)
    out = np.zeros((B, H, Lq, D), dtype=np.float64)
    _check(lib.oracle_prefill(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                              B, H, Lq, D, bs, nb, bt.shape[1], float(scale),
                              _ptr(out)))
    return out


def prefill_varlen(q, k_cache, v_cache, block_tables, context_lens, q_lens, scale, lib=None):
    """Chunks of different lengths: q[B,H,Lq,D] fp16 holds sequence b's
    q_lens[b] new queries in rows 0 .. q_lens[b]-1 (the last q_lens[b]
    positions of its context, end-aligned causal mask).  Each sequence is
    the fixed-length prefill of its own rows; rows past q_lens[b] are zero.
    -> out[B,H,Lq,D] fp64."""
    qb = _bits(q)
    B, H, Lq, D = qb.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(B, -1)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32).reshape(B)
    ql = np.ascontiguousarray(q_lens, dtype=np.int64).reshape(B)
    if np.any(ql < 0) or np.any(ql > Lq) or np.any(ql > cl):
        raise OracleError(3)
    out = np.zeros((B, H, Lq, D), dtype=np.float64)
    for b in range(B):
        n = int(ql[b])
        if n > 0:
            out[b:b + 1, :, :n] = prefill(qb[b:b + 1, :, :n], k_cache, v_cache, bt[b:b + 1],
                                          cl[b:b + 1], scale, lib)
    return out


def kv_cache_write(k, v, slot_mapping, k_cache, v_cache, lib=None):
    """Returns new (k_cache, v_cache) as uint16 bit arrays; inputs untouched."""
    lib = lib or load()
    kb, vb = _bits(k), _bits(v)
    T, H, D = kb.shape
    kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
    nb, bs = kc.shape[0], kc.shape[1]
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64).reshape(T)
    _check(lib.oracle_kv_cache_write(_ptr(kb), _ptr(vb), _ptr(sm), T, H, D, bs,
                                     nb, _ptr(kc), _ptr(vc)))
    return kc, vc


def block_copy(k_cache, v_cache, pairs, lib=None):
    """pairs[N,2] (src, dst).  Returns new (k_cache, v_cache) bit arrays."""
    lib = lib or load()
    kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
    nb, bs, H, D = kc.shape
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    _check(lib.oracle_block_copy(_ptr(kc), _ptr(vc), _ptr(pr), pr.shape[0], H,
                                 D, bs, nb))
    return kc, vc


def gather(pool, table, seq_len, head, lib=None):
    """Contiguous fp64 [seq_len, D] copy of one head's keys (or values)."""
    lib = lib or load()
    pb = _bits(pool)
    nb, bs, H, D = pb.shape
    tb = np.ascontiguousarray(table, dtype=np.int32)
    out = np.zeros((seq_len, D), dtype=np.float64)
    _check(lib.oracle_gather(_ptr(pb), _ptr(tb), int(tb.size), int(seq_len), H,
                             int(head), D, bs, nb, _ptr(out)))
    return out


def e4m3_to_double(code, lib=None):
    lib = lib or load()
    return lib.oracle_e4m3_to_double(int(code) & 0xFF)


def e4m3_from_float(x, lib=None):
    lib = lib or load()
    return lib.oracle_e4m3_from_float(float(np.float32(x)))


def kv_cache_write_fp8(k, v, slot_mapping, k8, v8, kscale, vscale, lib=None):
    """Quantizing cache write.  k, v [T,H,D] fp16; k8/v8 [NB,bs,H,D] uint8;
    kscale/vscale [NB,H,bs] float32.  Returns new (k8, v8, kscale, vscale)."""
    lib = lib or load()
    kb, vb = _bits(k), _bits(v)
    T, H, D = kb.shape
    k8 = np.ascontiguousarray(k8, dtype=np.uint8).copy()
    v8 = np.ascontiguousarray(v8, dtype=np.uint8).copy()
    ks = np.ascontiguousarray(kscale, dtype=np.float32).copy()
    vs = np.ascontiguousarray(vscale, dtype=np.float32).copy()
    nb, bs = k8.shape[0], k8.shape[1]
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64).reshape(T)
    _check(lib.oracle_kv_cache_write_fp8(_ptr(kb), _ptr(vb), _ptr(sm), T, H, D, bs, nb,
                                         _ptr(k8), _ptr(v8), _ptr(ks), _ptr(vs)))
    return k8, v8, ks, vs


def decode_fp8(q, k8, v8, kscale, vscale, block_tables, context_lens, scale, lib=None):
    """Decode over an e4m3 cache (exact dequantization): out[B,H,D] fp64."""
    lib = lib or load()
    qb = _bits(q)
    B, H, D = qb.shape
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    v8 = np.ascontiguousarray(v8, dtype=np.uint8)
    ks = np.ascontiguousarray(kscale, dtype=np.float32)
    vs = np.ascontiguousarray(vscale, dtype=np.float32)
    nb, bs = k8.shape[0], k8.shape[1]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(B, -1)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32).reshape(B)
    out = np.zeros((B, H, D), dtype=np.float64)
    _check(lib.oracle_decode_fp8(_ptr(qb), _ptr(k8), _ptr(v8), _ptr(ks), _ptr(vs), _ptr(bt),
                                 _ptr(cl), B, H, D, bs, nb, bt.shape[1], float(scale),
                                 _ptr(out)))
    return out
