"""GB300-native paged-KV attention: ctypes binding of libpagedkv.

The compute path is the C-ABI CUDA library (include/pagedkv.h, sources in
csrc/); this package only marshals torch tensors into it.  Importing the
package does not load the library; the first call does, and raises if the
library has not been built (``build_lib.build()``).
"""
from ._lib import (  # noqa: F401
    EXPORTS, LIB_PATH, PA_DEV_BAD_BLOCK_ID, PA_DEV_BAD_CONTEXT, PA_DEV_BAD_PAIR,
    PA_DEV_BAD_SLOT, PA_DEV_TIMEOUT, PA_ERR_CUDA, PA_ERR_INVALID, PA_ERR_UNSUPPORTED,
    PA_ERR_WORKSPACE, PA_OK, PagedKVError, host_device_pointer, lib, pa_block_copy, pa_decode,
    pa_decode_append,
    pa_decode_partition_tokens, pa_decode_shared_prefix, pa_decode_workspace_size,
    pa_shared_prefix_groups, pa_kv_cache_write, pa_kv_cache_write_fp8, pa_decode_fp8,
    pa_prefill_chunk, pa_prefill_chunk_varlen, pa_prefill_workspace_size, status_string,
)
