"""CSA / HCA hybrid compressed attention for B300 (sm_103a).

Thin Python binding over the C ABI of include/csa.h (libcsa_b300.so, built in-tree by
`python -m long_context_compressed_pooling_b300.build`). It only marshals torch tensors into
pointers and sizes, allocates workspaces with torch, and passes torch's current CUDA stream;
every step of the computation runs in the library's CUDA kernels. The library is loaded on the
first call; that call raises when it is missing, and every call refuses host tensors: there is
no CPU or fallback path.
"""
from ._native import (  # noqa: F401
    CSA_OK,
    CsaError,
    FAULT_SKIP_KEY_COPIES,
    LIB_PATH,
    MAX_COPIES,
    PAGE_TOKENS,
    PreparedLayerPair,
    PreparedPagedPair,
    PreparedPagedStep,
    RING_TOKENS,
    compress,
    compress_index_keys,
    csa_attend,
    device_status,
    exported_symbols,
    hca_attend,
    index_scores,
    index_topk,
    layer_pair,
    lse_merge,
    load_library,
    scatter_rows,
    paged_decode_step,
    profiler_collect,
    profiler_enable,
    quantize_mxfp4,
    shard_candidates,
    test_set_faults,
    topk,
    topk_f32,
    topk_merge,
    workspace_sizes,
)
