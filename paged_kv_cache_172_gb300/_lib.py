"""ctypes binding of libpagedkv (include/pagedkv.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  If the compiled
library is missing the first call raises; there is no fallback.
"""
import ctypes
import functools
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)
PA_DEV_BAD_BLOCK_ID = 0x1
PA_DEV_BAD_CONTEXT = 0x2
PA_DEV_BAD_SLOT = 0x4
PA_DEV_BAD_PAIR = 0x8
PA_DEV_TIMEOUT = 0x10

# Every symbol include/pagedkv.h declares.
EXPORTS = (
    "pa_status_string", "pa_last_cuda_error", "pa_version", "pa_host_device_pointer",
    "pa_decode_partition_tokens", "pa_decode_workspace_size", "pa_decode",
    "pa_prefill_workspace_size", "pa_prefill_chunk", "pa_prefill_chunk_varlen",
    "pa_kv_cache_write", "pa_block_copy",
    "pa_decode_static",
    "pa_decode_append", "pa_decode_shared_prefix", "pa_shared_prefix_groups",
    "pa_kv_cache_write_fp8", "pa_decode_fp8",
)

# Size of the fixed scratch array behind pa_decode_static (PA_DECODE_STATIC_SCRATCH_BYTES).
PA_DECODE_STATIC_SCRATCH_BYTES = 8 << 20


class PagedKVError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {status_string(code)}")


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def _bind(lib):
    lib.pa_status_string.argtypes = [_I]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_cuda_error.argtypes = []
    lib.pa_last_cuda_error.restype = _I
    lib.pa_version.argtypes = []
    lib.pa_version.restype = _I
    lib.pa_host_device_pointer.argtypes = [_P, ctypes.POINTER(ctypes.c_void_p)]
    lib.pa_host_device_pointer.restype = _I
    lib.pa_decode_partition_tokens.argtypes = [_I, _I, _I, _I]
    lib.pa_decode_partition_tokens.restype = _I
    lib.pa_decode_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
    lib.pa_decode_workspace_size.restype = _SZ
    lib.pa_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                              ctypes.c_float, _P, _P, _SZ, _P, _P]
    lib.pa_decode.restype = _I
    lib.pa_prefill_workspace_size.argtypes = [_I, _I, _I, _I]
    lib.pa_prefill_workspace_size.restype = _SZ
    lib.pa_prefill_chunk.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _P, _P, _SZ, _P, _P]
    lib.pa_prefill_chunk.restype = _I
    lib.pa_prefill_chunk_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                            ctypes.c_float, _P, _P, _SZ, _P, _P]
    lib.pa_prefill_chunk_varlen.restype = _I
    lib.pa_kv_cache_write.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]
    lib.pa_kv_cache_write.restype = _I
    lib.pa_block_copy.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]
    lib.pa_block_copy.restype = _I
    lib.pa_decode_static.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _P, _P, _P]
    lib.pa_decode_static.restype = _I
    lib.pa_decode_append.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _P, _P, _SZ, _P, _P]
    lib.pa_decode_append.restype = _I
    lib.pa_decode_shared_prefix.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                            _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                                            _SZ, _P, _P]
    lib.pa_decode_shared_prefix.restype = _I
    lib.pa_shared_prefix_groups.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                            ctypes.POINTER(_I)]
    lib.pa_shared_prefix_groups.restype = _I
    lib.pa_kv_cache_write_fp8.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    lib.pa_kv_cache_write_fp8.restype = _I
    lib.pa_decode_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                  ctypes.c_float, _P, _P, _SZ, _P, _P]
    lib.pa_decode_fp8.restype = _I
    return lib


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libpagedkv.so not found at {LIB_PATH}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(code):
    return lib().pa_status_string(int(code)).decode()


def _check(rc, what):
    if rc != PA_OK:
        err = PagedKVError(rc, what)
        if rc == PA_ERR_CUDA:
            err.cuda_error = lib().pa_last_cuda_error()
        raise err


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def host_device_pointer(t):
    """Device address of a pinned CPU tensor's data (pa_host_device_pointer):
    a kernel given it loads and stores the host memory directly."""
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("host_device_pointer takes a CPU tensor")
    d = ctypes.c_void_p()
    _check(lib().pa_host_device_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(d)),
           "pa_host_device_pointer")
    return d.value


def _io(t, dtype, name, ndim):
    """Pointer for a per-call input or output that the kernel may access in
    place: a CUDA tensor, or a pinned CPU tensor (its mapped device address)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous() or t.dim() != ndim:
            raise ValueError(f"{name} must be contiguous with {ndim} dims")
        return ctypes.c_void_p(host_device_pointer(t))
    _need(t, dtype, name, ndim)
    return _ptr(t)


def _one_device(fn):
    """All CUDA tensors and streams of a call on one device, and the call made
    with that device current: the library sets up and launches its kernels on
    the current device."""
    @functools.wraps(fn)
    def call(*args, **kwargs):
        devs = set()
        for a in list(args) + list(kwargs.values()):
            if isinstance(a, torch.Tensor) and a.is_cuda:
                devs.add(a.device)
            elif isinstance(a, torch.cuda.Stream):
                devs.add(a.device)
        if len(devs) > 1:
            raise ValueError(f"{fn.__name__}: CUDA tensors or streams on different devices: "
                             + ", ".join(sorted(str(d) for d in devs)))
        if devs:
            dev = devs.pop()
            if torch.cuda.current_device() != dev.index:
                with torch.cuda.device(dev):
                    return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return call


def pa_decode_partition_tokens(B, H, block_size, max_context_len):
    return lib().pa_decode_partition_tokens(B, H, block_size, max_context_len)


def pa_decode_workspace_size(B, H, D, block_size, max_context_len, partition_tokens=0):
    return lib().pa_decode_workspace_size(B, H, D, block_size, max_context_len,
                                          partition_tokens)


@_one_device
def pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
              out=None, partition_tokens=0, workspace=None, status=None, stream=None):
    """Paged decode attention.  q [B,H,D] fp16; caches [NB,bs,H,D] fp16;
    block_tables [B,max_blocks] int32; context_lens [B] int32;
    ``max_context_len`` is a host-side upper bound on context_lens.
    q, out, block_tables and context_lens may be pinned CPU tensors, read
    and written by the kernels in place.  Returns ``out`` [B,H,D] fp16
    (allocated on the device when not given)."""
    qp = _io(q, torch.float16, "q", 3)
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    btp = _io(block_tables, torch.int32, "block_tables", 2)
    clp = _io(context_lens, torch.int32, "context_lens", 1)
    B, H, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    if tuple(k_cache.shape) != (NB, bs, H, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, block_size, H, D]")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables/context_lens batch mismatch")
    dev = k_cache.device
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float16, device=dev)
    op = _io(out, torch.float16, "out", 3)
    ws_bytes = pa_decode_workspace_size(B, H, D, bs, max(int(max_context_len), 1),
                                        partition_tokens)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pa_decode(qp, _ptr(k_cache), _ptr(v_cache), btp, clp, B, H, D, bs, NB,
                         block_tables.shape[1],
                         int(max_context_len), int(partition_tokens), float(scale), op,
                         _ptr(workspace), ws_len, _ptr(status), _stream(stream, dev))
    _check(rc, "pa_decode")
    return out


@_one_device
def pa_decode_append(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                     max_context_len, out=None, partition_tokens=0, workspace=None, status=None,
                     stream=None):
    """Store each sequence's new token k_new/v_new [B,H,D] at position ctx-1
    of the paged cache and run decode attention including it (one launch).
    q, k_new, v_new, out, block_tables and context_lens may be pinned CPU
    tensors, read and written by the kernels in place.  Returns ``out``
    [B,H,D] fp16 (allocated on the device when not given)."""
    qp = _io(q, torch.float16, "q", 3)
    kp = _io(k_new, torch.float16, "k_new", 3)
    vp = _io(v_new, torch.float16, "v_new", 3)
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    btp = _io(block_tables, torch.int32, "block_tables", 2)
    clp = _io(context_lens, torch.int32, "context_lens", 1)
    B, H, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    if k_new.shape != q.shape or v_new.shape != q.shape:
        raise ValueError("k_new/v_new must be [B, H, D] like q")
    if tuple(k_cache.shape) != (NB, bs, H, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, block_size, H, D]")
    dev = k_cache.device
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float16, device=dev)
    op = _io(out, torch.float16, "out", 3)
    ws_bytes = pa_decode_workspace_size(B, H, D, bs, max(int(max_context_len), 1),
                                        partition_tokens)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_append(qp, kp, vp, _ptr(k_cache), _ptr(v_cache), btp, clp,
                                B, H, D, bs, NB,
                                block_tables.shape[1], int(max_context_len),
                                int(partition_tokens), float(scale), op, _ptr(workspace),
                                ws_len, _ptr(status), _stream(stream, dev))
    _check(rc, "pa_decode_append")
    return out


@_one_device
def pa_decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, seq_group,
                            group_offsets, group_seqs, group_prefix_len, scale, max_context_len,
                            max_group_size, max_prefix_len, out=None, partition_tokens=0,
                            workspace=None, status=None, stream=None):
    """Decode where groups of sequences share prefix blocks (CSR groups:
    members group_seqs[group_offsets[g]:group_offsets[g+1]], shared tokens
    group_prefix_len[g], seq_group[b] = group or -1; all int32 on device).
    Same result as pa_decode; shared partitions are read once per group."""
    _need(q, torch.float16, "q", 3)
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                    ("seq_group", seq_group), ("group_offsets", group_offsets),
                    ("group_seqs", group_seqs), ("group_prefix_len", group_prefix_len)):
        _need(t, torch.int32, name)
    B, H, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    G = group_prefix_len.numel()
    if group_offsets.numel() != G + 1 or seq_group.numel() != B:
        raise ValueError("group_offsets must have G+1 entries and seq_group B entries")
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = pa_decode_workspace_size(B, H, D, bs, max(int(max_context_len), 1),
                                        partition_tokens)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_shared_prefix(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(seq_group), _ptr(group_offsets), _ptr(group_seqs), _ptr(group_prefix_len), G,
        int(max_group_size), int(max_prefix_len), B, H, D, bs, NB, block_tables.shape[1],
        int(max_context_len), int(partition_tokens), float(scale), _ptr(out), _ptr(workspace),
        ws_len, _ptr(status), _stream(stream, q.device))
    _check(rc, "pa_decode_shared_prefix")
    return out


def pa_shared_prefix_groups(block_tables, context_lens, block_size, min_shared_tokens=0,
                            max_group_size=16):
    """Groups of sequences sharing leading physical blocks, from the block
    tables (host-side prefix tree).  Takes CPU or CUDA int32 tensors, returns
    CPU int32 tensors (seq_group [B], group_offsets [G+1], group_seqs [n],
    group_prefix_len [G]) in the form pa_decode_shared_prefix takes."""
    bt = block_tables.detach().to("cpu", torch.int32).contiguous()
    cl = context_lens.detach().to("cpu", torch.int32).contiguous()
    if bt.dim() != 2 or cl.dim() != 1 or cl.numel() != bt.shape[0]:
        raise ValueError("block_tables must be [B, max_blocks_per_seq] and context_lens [B]")
    B, M = bt.shape
    seq_group = torch.empty(B, dtype=torch.int32)
    offsets = torch.empty(B // 2 + 1, dtype=torch.int32)
    seqs = torch.empty(max(B, 1), dtype=torch.int32)
    plen = torch.empty(max(B // 2, 1), dtype=torch.int32)
    G = _I(0)
    rc = lib().pa_shared_prefix_groups(_ptr(bt), _ptr(cl), B, max(M, 1), int(block_size),
                                       int(min_shared_tokens), int(max_group_size),
                                       _ptr(seq_group), _ptr(offsets), _ptr(seqs), _ptr(plen),
                                       ctypes.byref(G))
    _check(rc, "pa_shared_prefix_groups")
    G = G.value
    offsets = offsets[:G + 1].clone()
    return seq_group, offsets, seqs[:int(offsets[-1])].clone(), plen[:G].clone()


@_one_device
def pa_kv_cache_write_fp8(k, v, slot_mapping, k_cache8, v_cache8, k_scale, v_scale, status=None,
                          stream=None):
    """Quantize k/v [T,H,D] fp16 into e4m3 pools k_cache8/v_cache8
    [NB,bs,H,D] uint8 with per-(token, head) scales k_scale/v_scale
    [NB,H,bs] float32, at slot_mapping [T] int64."""
    _need(k, torch.float16, "k", 3)
    _need(v, torch.float16, "v", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(k_cache8, torch.uint8, "k_cache8", 4)
    _need(v_cache8, torch.uint8, "v_cache8", 4)
    _need(k_scale, torch.float32, "k_scale", 3)
    _need(v_scale, torch.float32, "v_scale", 3)
    T, H, D = k.shape
    NB, bs = k_cache8.shape[0], k_cache8.shape[1]
    if tuple(k_scale.shape) != (NB, H, bs) or v_scale.shape != k_scale.shape:
        raise ValueError("scales must be [num_blocks, H, block_size]")
    rc = lib().pa_kv_cache_write_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), T, H, D, bs, NB,
                                     _ptr(k_cache8), _ptr(v_cache8), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(status), _stream(stream, k.device))
    _check(rc, "pa_kv_cache_write_fp8")


@_one_device
def pa_decode_fp8(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, context_lens, scale,
                  max_context_len, out=None, partition_tokens=0, workspace=None, status=None,
                  stream=None):
    """Paged decode over e4m3 pools with per-(token, head) scales."""
    _need(q, torch.float16, "q", 3)
    _need(k_cache8, torch.uint8, "k_cache8", 4)
    _need(v_cache8, torch.uint8, "v_cache8", 4)
    _need(k_scale, torch.float32, "k_scale", 3)
    _need(v_scale, torch.float32, "v_scale", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    B, H, D = q.shape
    NB, bs = k_cache8.shape[0], k_cache8.shape[1]
    if tuple(k_cache8.shape) != (NB, bs, H, D) or v_cache8.shape != k_cache8.shape:
        raise ValueError("fp8 pools must be [num_blocks, block_size, H, D]")
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = pa_decode_workspace_size(B, H, D, bs, max(int(max_context_len), 1),
                                        partition_tokens)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_fp8(_ptr(q), _ptr(k_cache8), _ptr(v_cache8), _ptr(k_scale),
                             _ptr(v_scale), _ptr(block_tables), _ptr(context_lens), B, H, D, bs,
                             NB, block_tables.shape[1], int(max_context_len),
                             int(partition_tokens), float(scale), _ptr(out), _ptr(workspace),
                             ws_len, _ptr(status), _stream(stream, q.device))
    _check(rc, "pa_decode_fp8")
    return out


def pa_prefill_workspace_size(B, H, Lq, D):
    """Bytes of workspace pa_prefill_chunk uses to split the grid's last round
    (0 when it needs none) on the current device."""
    return int(lib().pa_prefill_workspace_size(int(B), int(H), int(Lq), int(D)))


@_one_device
def pa_prefill_chunk(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                     workspace=None, tail_split=True, status=None, stream=None, q_lens=None):
    """Chunked prefill attention.  q [B,H,Lq,D] fp16 are the last Lq positions
    of each sequence (end-aligned causal mask).  Returns out [B,H,Lq,D].
    With q_lens ([B] int32 on the device), sequence b has q_lens[b] <= Lq new
    queries in rows 0 .. q_lens[b]-1 and its later rows of out are zeros
    (pa_prefill_chunk_varlen).  A workspace for the tail split is allocated
    when not given; tail_split=False passes none (every work unit runs whole)."""
    _need(q, torch.float16, "q", 4)
    if q_lens is not None:
        _need(q_lens, torch.int32, "q_lens", 1)
        if q_lens.numel() != q.shape[0]:
            raise ValueError("q_lens must have one entry per sequence")
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    B, H, Lq, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    if tuple(k_cache.shape) != (NB, bs, H, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, block_size, H, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, torch.float16, "out", 4)
    if not tail_split:
        workspace = None
    elif workspace is None:
        ws_bytes = pa_prefill_workspace_size(B, H, Lq, D) if B * Lq > 0 else 0
        if ws_bytes > 0:
            workspace = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if q_lens is None:
        rc = lib().pa_prefill_chunk(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                    _ptr(context_lens), B, H, Lq, D, bs, NB,
                                    block_tables.shape[1], float(scale), _ptr(out),
                                    _ptr(workspace), ws_len, _ptr(status),
                                    _stream(stream, q.device))
        _check(rc, "pa_prefill_chunk")
    else:
        rc = lib().pa_prefill_chunk_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(block_tables), _ptr(context_lens), _ptr(q_lens),
                                           B, H, Lq, D, bs, NB, block_tables.shape[1],
                                           float(scale), _ptr(out), _ptr(workspace), ws_len,
                                           _ptr(status), _stream(stream, q.device))
        _check(rc, "pa_prefill_chunk_varlen")
    return out


@_one_device
def pa_prefill_chunk_varlen(q, k_cache, v_cache, block_tables, context_lens, q_lens, scale,
                            out=None, workspace=None, tail_split=True, status=None,
                            stream=None):
    """Chunked prefill with a chunk length per sequence: q [B,H,Lq_max,D]
    holds sequence b's q_lens[b] new queries in rows 0 .. q_lens[b]-1;
    out rows past q_lens[b] are zeros."""
    return pa_prefill_chunk(q, k_cache, v_cache, block_tables, context_lens, scale, out=out,
                            workspace=workspace, tail_split=tail_split, status=status,
                            stream=stream, q_lens=q_lens)


@_one_device
def pa_kv_cache_write(k, v, slot_mapping, k_cache, v_cache, status=None, stream=None):
    """Scatter k/v [T,H,D] fp16 into the caches at slot_mapping [T] int64."""
    _need(k, torch.float16, "k", 3)
    _need(v, torch.float16, "v", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    T, H, D = k.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    if v.shape != k.shape or slot_mapping.shape[0] != T:
        raise ValueError("k/v/slot_mapping shape mismatch")
    if tuple(k_cache.shape) != (NB, bs, H, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, block_size, H, D]")
    rc = lib().pa_kv_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, H, D, bs, NB,
                                 _ptr(k_cache), _ptr(v_cache), _ptr(status),
                                 _stream(stream, k.device))
    _check(rc, "pa_kv_cache_write")


@_one_device
def pa_block_copy(k_cache, v_cache, pairs, status=None, stream=None):
    """Copy whole physical blocks: pairs [N,2] int64 (src, dst)."""
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    _need(pairs, torch.int64, "pairs", 2)
    NB, bs, H, D = k_cache.shape
    if v_cache.shape != k_cache.shape or pairs.shape[1] != 2:
        raise ValueError("bad k_cache/v_cache/pairs shapes")
    rc = lib().pa_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0], H, D,
                             bs, NB, _ptr(status), _stream(stream, k_cache.device))
    _check(rc, "pa_block_copy")
