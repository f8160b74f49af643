"""Hybrid-precision (4-bit + BF16) KV-cache attention for one GB300 GPU.

Python binding of libhyq (include/hyq.h).  The compute runs in the library's
hand-written CUDA kernels for sm_103a; PyTorch only provides device memory and
streams.  Build the library with ``__graft_entry__.build()``.
"""
from . import _lib
from ._lib import (HyqConfig, HyqError, HyqLayout, load, lib_path, hyq_config_check,
                   hyq_age_tail, hyq_decode_append, hyq_decode_attention, hyq_decode_step,
                   hyq_decode_step_prefetch,
                   hyq_decode_attention_noalloc, hyq_layout_reset, hyq_layout_sizes, hyq_prefill_attention,
                   hyq_prefill_attention_band,
                   hyq_quantize_append, hyq_read_device_error, hyq_rebuild, hyq_select_vertical,
                   hyq_select_vertical_heads, hyq_select_vertical_mass, hyq_set_decode_plan, hyq_set_decode_overlap,
                   hyq_status_string, hyq_vl_count, hyq_workspace_size)
from .cache import (HybridDecoder, HybridLayer, make_config, pack_qblocks, unpack_qblocks,
                    workspace)

__all__ = [n for n in dir() if not n.startswith("_")]
