"""Host-facing decode step: device-resident paged KV state, host I/O per step.

A serving loop keeps the KV pool, block tables and workspace on the GPU and
moves only each step's small inputs (queries, the new tokens' K/V, updated
lengths and tables) and the attention output across the host link.  ``DecodeSession.step_from_host`` does exactly that around one
library call: host->device copies, pa_decode_append (the new tokens' cache
write fused into decode), device->host copy of the output, all asynchronous
on one stream.  The new token of sequence b sits at position
context_lens[b] - 1, so the step's slots follow from the block tables.
"""
import torch

from . import _lib


class DecodeSession:
    def __init__(self, k_cache, v_cache, B, max_blocks_per_seq, max_context_len, scale,
                 partition_tokens=0):
        self.k_cache, self.v_cache = k_cache, v_cache
        NB, bs, H, D = k_cache.shape
        dev = k_cache.device
        self.B, self.H, self.D, self.bs = B, H, D, bs
        self.max_context_len = int(max_context_len)
        self.scale = float(scale)
        self.partition_tokens = int(partition_tokens)
        self.q = torch.empty((B, H, D), dtype=torch.float16, device=dev)
        self.out = torch.empty_like(self.q)
        self.k_new = torch.empty((B, H, D), dtype=torch.float16, device=dev)
        self.v_new = torch.empty_like(self.k_new)
        self.context_lens = torch.empty(B, dtype=torch.int32, device=dev)
        self.block_tables = torch.empty((B, max_blocks_per_seq), dtype=torch.int32, device=dev)
        ws = _lib.pa_decode_workspace_size(B, H, D, bs, self.max_context_len,
                                           self.partition_tokens)
        self.workspace = torch.empty(max(ws // 4, 1) + 4, dtype=torch.float32, device=dev)

    def host_buffers(self):
        """Pinned host tensors matching the per-step inputs and the output."""
        pin = dict(pin_memory=True)
        return {
            "q": torch.empty(self.q.shape, dtype=torch.float16, **pin),
            "k_new": torch.empty(self.k_new.shape, dtype=torch.float16, **pin),
            "v_new": torch.empty(self.v_new.shape, dtype=torch.float16, **pin),
            "context_lens": torch.empty(self.context_lens.shape, dtype=torch.int32, **pin),
            "block_tables": torch.empty(self.block_tables.shape, dtype=torch.int32, **pin),
            "out": torch.empty(self.out.shape, dtype=torch.float16, **pin),
        }

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in
                   (self.q, self.k_new, self.v_new, self.context_lens, self.block_tables))

    def d2h_bytes(self):
        return self.out.numel() * self.out.element_size()

    def step_from_host(self, host, status=None, stream=None):
        """One decode step from pinned host buffers (see host_buffers()); the
        output lands in host['out'] when the stream reaches the end."""
        for name, dst in (("q", self.q), ("k_new", self.k_new), ("v_new", self.v_new),
                          ("context_lens", self.context_lens),
                          ("block_tables", self.block_tables)):
            dst.copy_(host[name], non_blocking=True)
        _lib.pa_decode_append(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                              self.block_tables, self.context_lens, self.scale,
                              self.max_context_len, out=self.out,
                              partition_tokens=self.partition_tokens, workspace=self.workspace,
                              status=status, stream=stream)
        host["out"].copy_(self.out, non_blocking=True)
        return host["out"]
