"""ctypes binding of the C++ float64 oracle (``oracle/cpp/hyq_oracle.cpp``).

Test infrastructure, like the rest of ``oracle/``: only the tests, the
smoke check and the benchmark's CPU-baseline legs use it.  The C++ file is
an independent restatement of the same passages as the Python modules of
this package (the tests assert that the two agree), written in plain C++17
with float64 accumulation and its own binary16 / e4m3 arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpp", "hyq_oracle.cpp")
LIB = os.path.join(HERE, "cpp", "libhyq_oracle.so")

_lib = None
_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_i64_p = ctypes.POINTER(ctypes.c_int64)
_c_u8_p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle library with g++ (no fused multiply-add contraction)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", SRC, "-o", LIB]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"g++ failed:\n{' '.join(cmd)}\n{r.stderr}")
    return LIB


def load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB)
        lib.hyqo_quantize.restype = ctypes.c_int
        lib.hyqo_quantize.argtypes = [_c_double_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _c_u8_p,
                                      _c_double_p, _c_double_p]
        lib.hyqo_vl_count.restype = ctypes.c_int64
        lib.hyqo_vl_count.argtypes = [ctypes.c_int64, ctypes.c_int64]
        lib.hyqo_e4m3_value.restype = ctypes.c_double
        lib.hyqo_e4m3_value.argtypes = [ctypes.c_int]
        lib.hyqo_e2m1_value.restype = ctypes.c_double
        lib.hyqo_e2m1_value.argtypes = [ctypes.c_int]
        lib.hyqo_select.restype = ctypes.c_int64
        lib.hyqo_select.argtypes = [_c_double_p, _c_double_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int, _c_i64_p, _c_double_p, ctypes.c_int]
        lib.hyqo_select_heads.restype = ctypes.c_int64
        lib.hyqo_select_heads.argtypes = [_c_double_p, _c_double_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, _c_i64_p, _c_i64_p, _c_i64_p, ctypes.c_int]
        lib.hyqo_decode.restype = ctypes.c_int
        lib.hyqo_decode.argtypes = [_c_double_p, _c_double_p, _c_double_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _c_i64_p,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int, _c_double_p, ctypes.c_int]
        lib.hyqo_prefill.restype = None
        lib.hyqo_prefill.argtypes = [_c_double_p, _c_double_p, _c_double_p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int64, _c_i64_p,
                                     ctypes.c_int64, ctypes.c_int, ctypes.c_int, _c_u8_p, _c_u8_p, _c_double_p,
                                     _c_double_p, ctypes.c_int]
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a, t):
    return None if a is None else a.ctypes.data_as(t)


def quantize(x, bits: int = 4):
    """Codes uint8 [..., d], scale / zero float64 [..., d / 32]; raises on a range error."""
    x = _f64(x)
    d = x.shape[-1]
    n = x.size // d
    codes = np.zeros(x.shape, np.uint8)
    scale = np.zeros(x.shape[:-1] + (d // 32,))
    zero = np.zeros_like(scale)
    if load().hyqo_quantize(_p(x, _c_double_p), n, d, bits, _p(codes, _c_u8_p), _p(scale, _c_double_p),
                            _p(zero, _c_double_p)):
        raise ValueError("a group's step or zero is not a finite binary16")
    return codes, scale, zero


def vl_count(P: int, rho_ppm: int) -> int:
    return int(load().hyqo_vl_count(P, rho_ppm))


def e4m3_value(code: int) -> float:
    return float(load().hyqo_e4m3_value(code))


def e2m1_values() -> list:
    return [float(load().hyqo_e2m1_value(c)) for c in range(8)]


def select_vertical(q_proxy, k_src, L: int, window: int, rho_ppm: int, mass: bool = False, threads: int = 1):
    """(idx int64 [B, HKV, k] ascending, S float64 [B, HKV, P])."""
    q = _f64(q_proxy)
    k = _f64(k_src)
    B, HQ, T, d = q.shape
    HKV, ldk = k.shape[1], k.shape[2]
    P = max(0, L - window)
    kk = vl_count(P, rho_ppm)
    idx = np.zeros((B, HKV, kk), np.int64)
    S = np.zeros((B, HKV, P))
    load().hyqo_select(_p(q, _c_double_p), _p(k, _c_double_p), B, HQ, HKV, T, ldk, d, L, window, rho_ppm,
                       int(mass), _p(idx, _c_i64_p), _p(S, _c_double_p), threads)
    return idx, S


def select_vertical_heads(q_proxy, k_src, L: int, window: int, rho_ppm: int, threads: int = 1):
    """(idx_heads int64 [B, HQ, k], idx_kv int64 [B, HKV, ku], union sizes [B, HKV])."""
    q = _f64(q_proxy)
    k = _f64(k_src)
    B, HQ, T, d = q.shape
    HKV, ldk = k.shape[1], k.shape[2]
    P = max(0, L - window)
    kk = vl_count(P, rho_ppm)
    ku = min(P, (HQ // HKV) * kk)
    ih = np.zeros((B, HQ, kk), np.int64)
    ik = np.zeros((B, HKV, ku), np.int64)
    us = np.zeros((B, HKV), np.int64)
    load().hyqo_select_heads(_p(q, _c_double_p), _p(k, _c_double_p), B, HQ, HKV, T, ldk, d, L, window, rho_ppm,
                             _p(ih, _c_i64_p), _p(ik, _c_i64_p), _p(us, _c_i64_p), threads)
    return ih, ik, us


def hybrid_decode(q, k_src, v_src, L: int, P: int, idx, bits: int = 4, bits_v=None, threads: int = 0):
    """o [B, HQ, d] float64."""
    q = _f64(q)
    k = _f64(k_src)
    v = _f64(v_src)
    B, HQ, d = q.shape
    HKV, ldk = k.shape[1], k.shape[2]
    ix = np.zeros((B, HKV, 0), np.int64) if idx is None else np.ascontiguousarray(np.asarray(idx, np.int64))
    out = np.zeros((B, HQ, d))
    if load().hyqo_decode(_p(q, _c_double_p), _p(k, _c_double_p), _p(v, _c_double_p), B, HQ, HKV, ldk, d, L, P,
                          _p(ix, _c_i64_p), ix.shape[-1], bits, bits if bits_v is None else bits_v,
                          _p(out, _c_double_p), threads):
        raise ValueError("a group's step or zero is not a finite binary16")
    return out


def hybrid_prefill(q, k, v, vl_idx, window: int, dtype: str = "int8", query_blocks=None, heads=None,
                   band: bool = False, threads: int = 0):
    """(o, a) float64 [B, HQ, L, d]: the output and sum_j p_j |v_j| / sum_j p_j."""
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    B, HQ, L, d = q.shape
    HKV = k.shape[1]
    ix = np.zeros((B, HKV, 0), np.int64) if vl_idx is None else np.ascontiguousarray(np.asarray(vl_idx, np.int64))
    nblk = -(-L // 128)
    bm = None if query_blocks is None else np.isin(np.arange(nblk), query_blocks).astype(np.uint8)
    hm = None if heads is None else np.isin(np.arange(HQ), heads).astype(np.uint8)
    out = np.zeros(q.shape)
    mag = np.zeros(q.shape)
    load().hyqo_prefill(_p(q, _c_double_p), _p(k, _c_double_p), _p(v, _c_double_p), B, HQ, HKV, L, d, window,
                        _p(ix, _c_i64_p), ix.shape[-1], {"int8": 1, "fp8": 2, "fp4": 3}[dtype], int(band), _p(bm, _c_u8_p),
                        _p(hm, _c_u8_p), _p(out, _c_double_p), _p(mag, _c_double_p), threads)
    return out, mag
