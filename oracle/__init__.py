"""The fp64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports it and shares no code with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision, plain
loops, OpenMP across (sequence, head) units only).  This module compiles it with
gcc on first use and wraps it with ctypes, taking and returning numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# No -ffast-math: sums are never re-associated.  -ffp-contract=off keeps a*b+c
# as two roundings on every architecture (gcc on Arm would fuse it otherwise).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]
_lock = threading.Lock()


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
            return out
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-I", os.path.dirname(src), src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        return out


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes wrapper around one build of ``pkv_oracle.c``."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_slot_mapping.argtypes = [vp, vp, i64, vp, vp, i64, i32]
        lib.oracle_slot_mapping.restype = i32
        lib.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32]
        lib.oracle_reshape_and_cache.restype = i32
        lib.oracle_paged_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                               i32, i64, dbl, i32, vp]
        lib.oracle_paged_attention.restype = i32
        lib.oracle_copy_blocks.argtypes = [vp, vp, vp, i64, i64, i64]
        lib.oracle_copy_blocks.restype = i32
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = dbl
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                                     ctypes.c_float, ctypes.c_float]
        lib.oracle_reshape_and_cache_fp8.restype = i32
        lib.oracle_paged_attention_fp8.argtypes = [vp, vp, vp, vp, dbl, dbl, vp, vp, vp, i64, i64, i32,
                                                   i32, i32, i32, i64, dbl, i32, vp]
        lib.oracle_paged_attention_fp8.restype = i32
        self.lib = lib

    # -- threads ---------------------------------------------------------------
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))

    # -- step a1: slot mapping -------------------------------------------------
    def slot_mapping(self, block_tables, token_seq, token_pos, block_size: int) -> np.ndarray:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        ts = np.ascontiguousarray(token_seq, dtype=np.int32)
        tp = np.ascontiguousarray(token_pos, dtype=np.int32)
        out = np.empty(ts.shape[0], dtype=np.int64)
        rc = self.lib.oracle_slot_mapping(_p(out), _p(bt), bt.shape[1], _p(ts), _p(tp), ts.shape[0],
                                          block_size)
        if rc != 0:
            raise ValueError("oracle_slot_mapping: invalid input")
        return out

    # -- step a2: KV write -----------------------------------------------------
    def reshape_and_cache(self, k_cache, v_cache, k, v, slot_mapping) -> None:
        """Writes into k_cache/v_cache (uint16 [NB, bs, Hkv, d]) in place."""
        assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
        assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
        NB, bs, Hkv, d = k_cache.shape
        kk = np.ascontiguousarray(k, dtype=np.uint16)
        vv = np.ascontiguousarray(v, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        rc = self.lib.oracle_reshape_and_cache(_p(k_cache), _p(v_cache), _p(kk), _p(vv), _p(sm),
                                               sm.shape[0], NB, bs, Hkv, d)
        if rc != 0:
            raise ValueError("oracle_reshape_and_cache: slot outside the pool")

    # -- steps a3-a8: attention over the paged cache ----------------------------
    def paged_attention(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                        query_start_loc=None, causal: bool = True, row_mask=None) -> np.ndarray:
        """Returns fp64 [total_q, Hq, d]; rows outside ``row_mask`` are NaN."""
        qq = np.ascontiguousarray(q, dtype=np.uint16)
        total_q, Hq, d = qq.shape
        NB, bs, Hkv, d2 = k_cache.shape
        assert d2 == d
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        qsl = None if query_start_loc is None else np.ascontiguousarray(query_start_loc, np.int32)
        rm = None if row_mask is None else np.ascontiguousarray(row_mask, dtype=np.uint8)
        out = np.full((total_q, Hq, d), np.nan, dtype=np.float64)
        rc = self.lib.oracle_paged_attention(
            _p(out), _p(qq), _p(np.ascontiguousarray(k_cache)), _p(np.ascontiguousarray(v_cache)),
            _p(bt), _p(cl), _p(qsl), cl.shape[0], bt.shape[1], Hq, Hkv, d, bs, NB, float(scale),
            int(bool(causal)), _p(rm))
        if rc != 0:
            raise ValueError("oracle_paged_attention: invalid input")
        return out


    # -- copy-on-write block copy -----------------------------------------------
    def copy_blocks(self, k_cache, v_cache, pairs) -> None:
        """Copies whole blocks in place (any dtype; pairs int32 [n, 2] of (src, dst))."""
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        assert k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype
        pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        NB = k_cache.shape[0]
        block_bytes = k_cache.nbytes // NB if NB else 0
        rc = self.lib.oracle_copy_blocks(_p(k_cache), _p(v_cache), _p(pr), pr.shape[0], NB, block_bytes)
        if rc != 0:
            raise ValueError("oracle_copy_blocks: block id outside the pool")

    # -- FP8 (OCP e4m3) cache ---------------------------------------------------
    def e4m3_decode(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_decode(int(code) & 0xFF))

    def e4m3_encode(self, y: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(y)))

    def reshape_and_cache_fp8(self, k_cache, v_cache, k, v, slot_mapping, k_scale: float,
                              v_scale: float) -> None:
        """Writes e4m3 codes into k_cache/v_cache (uint8 [NB, bs, Hkv, d]) in place."""
        assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous
        assert v_cache.dtype == np.uint8 and v_cache.flags.c_contiguous
        NB, bs, Hkv, d = k_cache.shape
        kk = np.ascontiguousarray(k, dtype=np.uint16)
        vv = np.ascontiguousarray(v, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        rc = self.lib.oracle_reshape_and_cache_fp8(_p(k_cache), _p(v_cache), _p(kk), _p(vv), _p(sm),
                                                   sm.shape[0], NB, bs, Hkv, d, float(k_scale),
                                                   float(v_scale))
        if rc != 0:
            raise ValueError("oracle_reshape_and_cache_fp8: slot outside the pool or bad scale")

    def paged_attention_fp8(self, q, k_cache, v_cache, k_scale: float, v_scale: float, block_tables,
                            context_lens, scale: float, query_start_loc=None, causal: bool = True,
                            row_mask=None) -> np.ndarray:
        """Attention over an e4m3 cache (uint8 codes); fp64 [total_q, Hq, d]."""
        qq = np.ascontiguousarray(q, dtype=np.uint16)
        total_q, Hq, d = qq.shape
        NB, bs, Hkv, d2 = k_cache.shape
        assert d2 == d and k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        qsl = None if query_start_loc is None else np.ascontiguousarray(query_start_loc, np.int32)
        rm = None if row_mask is None else np.ascontiguousarray(row_mask, dtype=np.uint8)
        out = np.full((total_q, Hq, d), np.nan, dtype=np.float64)
        rc = self.lib.oracle_paged_attention_fp8(
            _p(out), _p(qq), _p(np.ascontiguousarray(k_cache)), _p(np.ascontiguousarray(v_cache)),
            float(k_scale), float(v_scale), _p(bt), _p(cl), _p(qsl), cl.shape[0], bt.shape[1], Hq, Hkv,
            d, bs, NB, float(scale), int(bool(causal)), _p(rm))
        if rc != 0:
            raise ValueError("oracle_paged_attention_fp8: invalid input")
        return out


_default: Oracle | None = None


def load() -> Oracle:
    """The oracle built from this package's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
