"""ctypes binding of libhyq (include/hyq.h).

Argument marshalling only: every function here converts torch tensors to
device pointers and calls the C entry point of the same name; all the work
runs in the library's CUDA kernels.  Loading fails loudly when the library is
missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB

c_int32 = ctypes.c_int32
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p

HYQ_OK = 0
STATUS = {0: "HYQ_OK", 1: "HYQ_ERR_INVALID_ARG", 2: "HYQ_ERR_UNSUPPORTED", 3: "HYQ_ERR_WORKSPACE",
          4: "HYQ_ERR_CAPACITY", 5: "HYQ_ERR_CUDA", 6: "HYQ_ERR_DEVICE"}
DEVERR_QUANT_RANGE = 0x1
DEVERR_COUNT = 0x2
DEVERR_INDEX = 0x4
DEVERR_SCORE = 0x8
DEVERR_TIMEOUT = 0x10

QBLOCK_ROWS = 64
QBLOCK_BYTES = 10240          # B_K = B_V = 4


def qtile_bytes(bits_k: int = 4, bits_v: int = 4) -> int:
    """Bytes of one 16-row quantised tile (include/hyq.h)."""
    return 256 * ((bits_k or 4) + (bits_v or 4)) + 512


def qblock_bytes(bits_k: int = 4, bits_v: int = 4) -> int:
    return 4 * qtile_bytes(bits_k, bits_v)
COUNTS = 8
CNT_NQ, CNT_NVL, CNT_NTAIL, CNT_LEN, CNT_RING_N, CNT_RING_POS = range(6)
LAYOUT_FIELDS = ("qblocks", "vl_k", "vl_v", "vl_idx", "tail_k", "tail_v", "q_ring", "counts", "err")
OP_SELECT, OP_DECODE, OP_PREFILL, OP_SELECT_MASS, OP_PREFILL_BAND = 1, 2, 3, 4, 5
PREFILL_INT8, PREFILL_FP8, PREFILL_FP4 = 1, 2, 3
VL_PER_KV_HEAD, VL_PER_QUERY_HEAD = 0, 1

# Every symbol include/hyq.h declares.
SYMBOLS = ("hyq_status_string", "hyq_config_check", "hyq_vl_count", "hyq_layout_sizes",
           "hyq_workspace_size", "hyq_layout_reset", "hyq_quantize_append",
           "hyq_select_vertical", "hyq_rebuild", "hyq_decode_append", "hyq_decode_attention",
           "hyq_decode_attention_noalloc", "hyq_read_device_error", "hyq_set_decode_plan",
           "hyq_prefill_attention", "hyq_decode_step", "hyq_set_decode_overlap",
           "hyq_decode_step_prefetch", "hyq_age_tail", "hyq_select_vertical_mass",
           "hyq_prefill_attention_band", "hyq_select_vertical_heads")
NOALLOC_SCRATCH_BYTES = 4 << 20


class HyqConfig(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("num_q_heads", c_int32), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("group", c_int32), ("window", c_int32),
                ("period", c_int32), ("rho_ppm", c_int32), ("capacity", c_int32),
                ("bits_k", c_int32), ("bits_v", c_int32), ("vl_mode", c_int32)]


class HyqLayout(ctypes.Structure):
    _fields_ = [(name, c_void_p) for name in LAYOUT_FIELDS]


class HyqError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


_lib = None


def lib_path() -> str:
    return os.environ.get("HYQ_LIB", LIB)


def load() -> ctypes.CDLL:
    """Load libhyq.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libhyq not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    sig = {
        "hyq_status_string": (ctypes.c_char_p, [c_int32]),
        "hyq_config_check": (c_int32, [P(HyqConfig)]),
        "hyq_vl_count": (c_int32, [P(HyqConfig), c_int32]),
        "hyq_layout_sizes": (c_int32, [P(HyqConfig), P(c_size_t)]),
        "hyq_workspace_size": (c_size_t, [P(HyqConfig), ctypes.c_int, c_int32]),
        "hyq_layout_reset": (c_int32, [P(HyqConfig), P(HyqLayout), c_void_p]),
        "hyq_quantize_append": (c_int32, [P(HyqConfig), c_void_p, c_void_p, c_int32, P(HyqLayout), c_void_p]),
        "hyq_select_vertical": (c_int32, [P(HyqConfig), c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                          c_int32, c_void_p, P(c_int32), c_void_p, c_size_t, c_void_p]),
        "hyq_select_vertical_mass": (c_int32, [P(HyqConfig), c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                               c_int32, c_void_p, P(c_int32), c_void_p, c_size_t, c_void_p]),
        "hyq_select_vertical_heads": (c_int32, [P(HyqConfig), c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                                c_int32, c_void_p, c_void_p, P(c_int32), P(c_int32), c_void_p,
                                                c_size_t, c_void_p]),
        "hyq_rebuild": (c_int32, [P(HyqConfig), c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                  P(HyqLayout), c_void_p]),
        "hyq_decode_append": (c_int32, [P(HyqConfig), c_void_p, c_void_p, c_void_p, P(HyqLayout),
                                        c_void_p, c_void_p, c_int32, c_void_p]),
        "hyq_decode_attention": (c_int32, [P(HyqConfig), c_void_p, P(HyqLayout), c_void_p, c_int32,
                                           c_void_p, c_size_t, c_void_p]),
        "hyq_decode_attention_noalloc": (c_int32, [P(HyqConfig), c_void_p, P(HyqLayout), c_void_p, c_int32,
                                                   c_void_p]),
        "hyq_read_device_error": (c_int32, [c_void_p, P(c_int32), c_void_p]),
        "hyq_set_decode_plan": (c_int32, [c_int32, c_int32]),
        "hyq_age_tail": (c_int32, [P(HyqConfig), P(HyqLayout), c_void_p]),
        "hyq_set_decode_overlap": (c_int32, [c_int32]),
        "hyq_decode_step": (c_int32, [P(HyqConfig), c_void_p, c_void_p, c_void_p, P(HyqLayout), c_void_p,
                                      c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
        "hyq_decode_step_prefetch": (c_int32, [P(HyqConfig), c_void_p, c_void_p, c_void_p, P(HyqLayout),
                                               P(HyqLayout), c_void_p, c_void_p, c_int32, c_void_p, c_int32,
                                               c_void_p, c_size_t, c_void_p]),
        "hyq_prefill_attention": (c_int32, [P(HyqConfig), c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                                            c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                                            c_void_p, c_size_t, c_void_p]),
        "hyq_prefill_attention_band": (c_int32, [P(HyqConfig), c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                                                 c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                                                 c_void_p, c_size_t, c_void_p]),
    }
    for name in SYMBOLS:
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = sig[name]
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != HYQ_OK:
        raise HyqError(fn, status)


def ptr(t) -> int | None:
    """Device (or host) address of a tensor, None for None."""
    return None if t is None else t.data_ptr()


def stream_ptr(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# --- thin wrappers, same names as the C entry points ------------------------

def hyq_status_string(status: int) -> str:
    return load().hyq_status_string(status).decode()


def hyq_config_check(cfg: HyqConfig) -> int:
    return load().hyq_config_check(ctypes.byref(cfg))


def hyq_vl_count(cfg: HyqConfig, P: int) -> int:
    return load().hyq_vl_count(ctypes.byref(cfg), P)


def hyq_layout_sizes(cfg: HyqConfig) -> list[int]:
    out = (c_size_t * len(LAYOUT_FIELDS))()
    _check("hyq_layout_sizes", load().hyq_layout_sizes(ctypes.byref(cfg), out))
    return list(out)


def hyq_workspace_size(cfg: HyqConfig, op: int, len_hint: int = 0) -> int:
    return load().hyq_workspace_size(ctypes.byref(cfg), op, len_hint)


def hyq_layout_reset(cfg, lay: HyqLayout, stream=None):
    _check("hyq_layout_reset", load().hyq_layout_reset(ctypes.byref(cfg), ctypes.byref(lay), stream_ptr(stream)))


def hyq_quantize_append(cfg, k_rows, v_rows, n_rows: int, lay: HyqLayout, stream=None):
    _check("hyq_quantize_append", load().hyq_quantize_append(
        ctypes.byref(cfg), ptr(k_rows), ptr(v_rows), n_rows, ctypes.byref(lay), stream_ptr(stream)))


def row_ld(t) -> int:
    """Leading dimension (rows per head) of a [B, H, rows, 128] view whose rows
    are dense 128-element vectors and whose heads are evenly strided."""
    if t.dim() != 4 or t.shape[3] != 128 or t.stride(3) != 1 or t.stride(2) != 128:
        raise ValueError("expected a [B, H, rows, 128] tensor with dense rows")
    if t.stride(1) % 128 or (t.shape[0] > 1 and t.stride(0) != t.shape[1] * t.stride(1)):
        raise ValueError("heads must be evenly strided")
    return t.stride(1) // 128


def hyq_select_vertical(cfg, q_proxy, n_proxy: int, k_src, L: int, idx_out, ws, stream=None) -> int:
    """q_proxy [B, HQ, T, 128] (a view; its first n_proxy rows are used);
    k_src [B, HKV, ld, 128]; idx_out int32 [B, HKV, k] contiguous."""
    k_out = c_int32(0)
    _check("hyq_select_vertical", load().hyq_select_vertical(
        ctypes.byref(cfg), ptr(q_proxy), n_proxy, row_ld(q_proxy), ptr(k_src), row_ld(k_src), L,
        ptr(idx_out), ctypes.byref(k_out), ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)))
    return k_out.value


def hyq_select_vertical_mass(cfg, q_proxy, n_proxy: int, k_src, L: int, idx_out, ws, stream=None) -> int:
    """As hyq_select_vertical with the softmax-mass score of Eq. 4; the
    workspace is workspace(cfg, OP_SELECT_MASS, L)."""
    k_out = c_int32(0)
    _check("hyq_select_vertical_mass", load().hyq_select_vertical_mass(
        ctypes.byref(cfg), ptr(q_proxy), n_proxy, row_ld(q_proxy), ptr(k_src), row_ld(k_src), L,
        ptr(idx_out), ctypes.byref(k_out), ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)))
    return k_out.value


def hyq_select_vertical_heads(cfg, q_proxy, n_proxy: int, k_src, L: int, idx_heads, idx_out, ws,
                              stream=None) -> tuple:
    """Algorithm 1 per query head (cfg.vl_mode = VL_PER_QUERY_HEAD):
    idx_heads int32 [B, HQ, k] contiguous or None, idx_out int32 [B, HKV, ku]
    contiguous.  Returns (k, ku)."""
    k_out, ku_out = c_int32(0), c_int32(0)
    _check("hyq_select_vertical_heads", load().hyq_select_vertical_heads(
        ctypes.byref(cfg), ptr(q_proxy), n_proxy, row_ld(q_proxy), ptr(k_src), row_ld(k_src), L,
        None if idx_heads is None else ptr(idx_heads), ptr(idx_out), ctypes.byref(k_out), ctypes.byref(ku_out),
        ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)))
    return k_out.value, ku_out.value


def hyq_rebuild(cfg, k_src, v_src, L: int, idx, k: int, lay: HyqLayout, stream=None):
    ld = row_ld(k_src)
    if row_ld(v_src) != ld:
        raise ValueError("k_src and v_src must share the leading dimension")
    _check("hyq_rebuild", load().hyq_rebuild(
        ctypes.byref(cfg), ptr(k_src), ptr(v_src), ld, L, ptr(idx), k,
        ctypes.byref(lay), stream_ptr(stream)))


def hyq_decode_append(cfg, q, k_new, v_new, lay: HyqLayout, k_src=None, v_src=None, stream=None):
    ld = row_ld(k_src) if k_src is not None else 0
    _check("hyq_decode_append", load().hyq_decode_append(
        ctypes.byref(cfg), ptr(q), ptr(k_new), ptr(v_new), ctypes.byref(lay), ptr(k_src), ptr(v_src),
        ld, stream_ptr(stream)))


def hyq_decode_attention(cfg, q, lay: HyqLayout, out, ws, len_hint: int = 0, stream=None):
    _check("hyq_decode_attention", load().hyq_decode_attention(
        ctypes.byref(cfg), ptr(q), ctypes.byref(lay), ptr(out), len_hint, ptr(ws),
        ws.numel() * ws.element_size(), stream_ptr(stream)))


def hyq_decode_step(cfg, q, k_new, v_new, lay: HyqLayout, out, ws, k_src=None, v_src=None, len_hint: int = 0,
                    stream=None):
    """Append this token (as hyq_decode_append) and attend over the cache
    including it (as hyq_decode_attention), in one launch."""
    ld = row_ld(k_src) if k_src is not None else 0
    _check("hyq_decode_step", load().hyq_decode_step(
        ctypes.byref(cfg), ptr(q), ptr(k_new), ptr(v_new), ctypes.byref(lay), ptr(k_src), ptr(v_src), ld,
        ptr(out), len_hint, ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)))


def hyq_age_tail(cfg, lay: HyqLayout, stream=None):
    """Frozen-mode maintenance: the tail rows older than the window go to the
    4-bit stream (quantised as by hyq_quantize_append), the last W stay."""
    _check("hyq_age_tail", load().hyq_age_tail(ctypes.byref(cfg), ctypes.byref(lay), stream_ptr(stream)))


def hyq_decode_step_prefetch(cfg, q, k_new, v_new, lay: HyqLayout, next_lay, out, ws, k_src=None, v_src=None,
                             len_hint: int = 0, stream=None):
    """hyq_decode_step that, once each block has read its share of ``lay``,
    asks L2 to prefetch the share of ``next_lay`` (the layout of the next
    decode call, or None for none) that the same block index will read."""
    ld = row_ld(k_src) if k_src is not None else 0
    _check("hyq_decode_step_prefetch", load().hyq_decode_step_prefetch(
        ctypes.byref(cfg), ptr(q), ptr(k_new), ptr(v_new), ctypes.byref(lay),
        ctypes.byref(next_lay) if next_lay is not None else None, ptr(k_src), ptr(v_src), ld,
        ptr(out), len_hint, ptr(ws), ws.numel() * ws.element_size(), stream_ptr(stream)))


def hyq_decode_attention_noalloc(cfg, q, lay: HyqLayout, out, len_hint: int = 0, stream=None):
    """Decode attention with the library's own fixed scratch (no workspace):
    for callers that cannot allocate device memory.  Calls that overlap on the
    GPU race on the shared scratch."""
    _check("hyq_decode_attention_noalloc", load().hyq_decode_attention_noalloc(
        ctypes.byref(cfg), ptr(q), ctypes.byref(lay), ptr(out), len_hint, stream_ptr(stream)))


def hyq_prefill_attention(cfg, dtype: int, q, k, v, L: int, vl_idx, kvl: int, out, ws, err=None,
                          stream=None):
    """q [B, HQ, ldq, 128]; k, v [B, HKV, ldk, 128] (bf16 views with dense
    rows); vl_idx int32 [B, HKV, kvl] contiguous (or None when kvl = 0);
    out bf16 [B, HQ, L, 128] contiguous; err int32 [1] device or None."""
    _prefill("hyq_prefill_attention", cfg, dtype, q, k, v, L, vl_idx, kvl, out, ws, err, stream)


def hyq_prefill_attention_band(cfg, dtype: int, q, k, v, L: int, vl_idx, kvl: int, out, ws, err=None,
                               stream=None):
    """As hyq_prefill_attention with the window taken per query: row i sees
    (i - W, i] in BF16; workspace is workspace(cfg, OP_PREFILL_BAND, L)."""
    _prefill("hyq_prefill_attention_band", cfg, dtype, q, k, v, L, vl_idx, kvl, out, ws, err, stream)


def _prefill(name, cfg, dtype, q, k, v, L, vl_idx, kvl, out, ws, err, stream):
    ldk = row_ld(k)
    if row_ld(v) != ldk:
        raise ValueError("k and v must share the leading dimension")
    _check(name, getattr(load(), name)(
        ctypes.byref(cfg), dtype, ptr(q), row_ld(q), ptr(k), ptr(v), ldk, L,
        ptr(vl_idx) if kvl > 0 else None, kvl, ptr(out), ptr(err), ptr(ws),
        ws.numel() * ws.element_size(), stream_ptr(stream)))


DECODE_PLAN_AUTO, DECODE_PLAN_DIRECT, DECODE_PLAN_CLUSTER, DECODE_PLAN_GLOBAL = range(4)


def hyq_set_decode_plan(merge: int, splits: int = 0):
    """Override the decode split / merge plan (process-wide); 0 = automatic."""
    _check("hyq_set_decode_plan", load().hyq_set_decode_plan(merge, splits))


def hyq_set_decode_overlap(enable: bool):
    """Programmatic dependent launch of decode calls (process-wide).  Only for
    streams where the kernel before each decode call does not write that
    call's layout (see include/hyq.h)."""
    _check("hyq_set_decode_overlap", load().hyq_set_decode_overlap(1 if enable else 0))


def hyq_read_device_error(err_dev, stream=None) -> int:
    host = c_int32(0)
    st = load().hyq_read_device_error(ptr(err_dev), ctypes.byref(host), stream_ptr(stream))
    if st not in (0, 6):
        raise HyqError("hyq_read_device_error", st)
    return host.value
