"""GB300-native KV-cache buffered copy: the data path of DejaVuLib.

"DejaVu: KV-Cache Streaming for Fast, Fault-Tolerant Generative LLM
Serving" (ICML 2024), §3: gather (pack) the many small, non-contiguous K/V
slices of a max-length-preallocated cache into one contiguous buffer, scatter
(unpack) such a buffer back, and on top of that swap microbatches to pinned
host memory, stream the prompt cache layer by layer, and keep a host-side
replica of decode deltas that a cache can be restored from.

All work runs in the hand-written sm_103a kernels of ``libdv.so`` behind the C
ABI of ``include/dv.h``; this package only marshals arguments (see
``kv_cache_streaming_gb300.dv``).  Importing it fails if ``libdv.so`` has not
been built (``python kv_cache_streaming_gb300/build.py``; the build script
runs by path, since importing this package needs the library).
"""
from .dv import (  # noqa: F401
    DV_MAX_BATCH, DV_OK, DV_ERR_INVALID_ARG, DV_ERR_RANGE, DV_ERR_BUFFER_TOO_SMALL,
    DV_ERR_MISALIGNED, DV_ERR_CUDA, DV_ERR_TIMEOUT, DV_ERR_UNSUPPORTED,
    DV_VARIANT_AUTO, DV_VARIANT_FLAT, DV_VARIANT_TILE, DV_VARIANT_TOKEN,
    DvError, Cache, Streamer, Fetcher, Replica, lib, library_path,
    HostBuffer, dv_host_alloc, dv_host_free, host_empty,
    dv_abi_version, dv_allocation_extent, dv_debug_fault, dv_staging_bytes, dv_kv_pack, dv_kv_unpack, dv_kv_unpack_records, dv_naive_gather, dv_swap_out, dv_swap_in,
    dv_swap_out_noalloc, DV_NOALLOC_STAGING_BYTES,
    dv_streamer_create, dv_stream_layer, dv_streamer_wait, dv_streamer_destroy,
    dv_fetcher_create, dv_fetch_layer, dv_fetcher_wait, dv_fetcher_destroy,
    dv_replica_create, dv_replica_append, dv_replica_append_streamed, dv_replica_restore,
    dv_replica_restore_batched,
    dv_replica_restore_fetched, dv_replica_restore_fetched_steps,
    dv_replica_truncate,
    dv_replica_info, dv_replica_destroy,
    Swapper, dv_swapper_create, dv_swapper_acquire, dv_swapper_prefetch, dv_swapper_release,
    dv_swapper_wait, dv_swapper_destroy,
    DeltaStreamer, dv_delta_streamer_create, dv_delta_stream, dv_delta_streamer_join,
    dv_delta_streamer_wait, dv_delta_streamer_destroy,
)
