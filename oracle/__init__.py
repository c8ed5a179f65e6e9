"""fp64 CPU oracle for the paged KV-cache hot path (ctypes wrapper around oracle.c).

TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's CPU-baseline arm may import
this package. It shares no code with the CUDA library and never calls it.

Every function takes numpy arrays: bf16 tensors as uint16 bit patterns, indices as int32, and
returns float64 results. The arithmetic itself lives in oracle.c, which cites the source pages.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def _ptr(a: Optional[np.ndarray], kind):
    if a is None:
        return ctypes.cast(None, kind)
    return a.ctypes.data_as(kind)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """One loaded copy of the oracle library (tests may load mutated copies side by side)."""

    def __init__(self, library: Optional[str] = None):
        if library is None:
            library = _build.LIBRARY
            if _build.needs_build():
                _build.build(quiet=True)
        self.path = library
        lib = ctypes.CDLL(os.path.abspath(library))
        lib.oracle_kv_store.restype = ctypes.c_int64
        lib.oracle_kv_store.argtypes = [_u16p, _u16p, _i32p, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _u16p,
                                        _u16p]
        lib.oracle_gather_head.restype = ctypes.c_int
        lib.oracle_gather_head.argtypes = [_u16p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, _i32p, ctypes.c_int32, ctypes.c_int32,
                                           _f64p]
        lib.oracle_paged_decode.restype = ctypes.c_int
        lib.oracle_paged_decode.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, _i32p, ctypes.c_int32,
                                            _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                            _f64p, ctypes.c_int32]
        lib.oracle_paged_prefill.restype = ctypes.c_int
        lib.oracle_paged_prefill.argtypes = [_u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_int32,
                                             _i32p, ctypes.c_int32, _u16p, _u16p, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_double, _f64p,
                                             ctypes.c_int32]
        lib.oracle_max_threads.restype = ctypes.c_int
        i64 = ctypes.c_int64
        lib.oracle_copy_blocks.restype = ctypes.c_int32
        lib.oracle_copy_blocks.argtypes = [_u16p, _u16p, ctypes.c_int32, i64, _i32p,
                                           ctypes.c_int32]
        lib.oracle_gather_blocks.restype = ctypes.c_int32
        lib.oracle_gather_blocks.argtypes = [_u16p, _u16p, ctypes.c_int32, i64, _i32p,
                                             ctypes.c_int32, _u16p, _u16p]
        lib.oracle_scatter_blocks.restype = ctypes.c_int32
        lib.oracle_scatter_blocks.argtypes = [_u16p, _u16p, _i32p, ctypes.c_int32, _u16p, _u16p,
                                              ctypes.c_int32, i64]
        lib.oracle_xxh64.restype = ctypes.c_uint64
        lib.oracle_xxh64.argtypes = [ctypes.c_char_p, ctypes.c_int64, ctypes.c_uint64]
        lib.oracle_block_hashes.restype = ctypes.c_int32
        lib.oracle_block_hashes.argtypes = [_i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.POINTER(ctypes.c_uint64)]
        self.lib = lib

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    # -- KV store -------------------------------------------------------------------------------
    def kv_store(self, k, v, slot_mapping, k_cache, v_cache):
        """Return (k_cache', v_cache', invalid_count); the inputs are not modified."""
        kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
        vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
        NB, BS, Hkv, D = kc.shape
        k = _c(k, np.uint16)
        v = _c(v, np.uint16)
        sm = _c(slot_mapping, np.int32)
        assert k.shape == (len(sm), Hkv, D) and v.shape == k.shape
        bad = self.lib.oracle_kv_store(_ptr(k, _u16p), _ptr(v, _u16p), _ptr(sm, _i32p), len(sm),
                                       NB, BS, Hkv, D, _ptr(kc, _u16p), _ptr(vc, _u16p))
        return kc, vc, int(bad)

    # -- Block-table walk -----------------------------------------------------------------------
    def gather_head(self, cache, bt_row, length: int, kv_head: int) -> np.ndarray:
        cache = _c(cache, np.uint16)
        NB, BS, Hkv, D = cache.shape
        bt_row = _c(bt_row, np.int32)
        out = np.zeros((length, D), dtype=np.float64)
        rc = self.lib.oracle_gather_head(_ptr(cache, _u16p), NB, BS, Hkv, D, _ptr(bt_row, _i32p),
                                         length, kv_head, _ptr(out, _f64p))
        if rc:
            raise IndexError("block table walk left the pool")
        return out

    # -- Decode ---------------------------------------------------------------------------------
    def paged_decode(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     num_threads: int = 0) -> np.ndarray:
        q = _c(q, np.uint16)
        kc = _c(k_cache, np.uint16)
        vc = _c(v_cache, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        B, Hq, D = q.shape
        NB, BS, Hkv, D2 = kc.shape
        assert D == D2 and Hq % Hkv == 0 and bt.shape[0] == B and cl.shape == (B,)
        out = np.zeros((B, Hq, D), dtype=np.float64)
        nt = num_threads or self.max_threads()
        rc = self.lib.oracle_paged_decode(_ptr(q, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p), NB,
                                          BS, Hkv, D, _ptr(bt, _i32p), bt.shape[1],
                                          _ptr(cl, _i32p), B, Hq, float(scale), _ptr(out, _f64p),
                                          nt)
        if rc:
            raise IndexError("block table walk left the pool")
        return out

    # -- Prefill --------------------------------------------------------------------------------
    def paged_prefill(self, q, k, v, cu_seqlens_q, cu_seqlens_k, block_tables, k_cache, v_cache,
                      scale: float, num_threads: int = 0) -> np.ndarray:
        q = _c(q, np.uint16)
        k = _c(k, np.uint16)
        v = _c(v, np.uint16)
        cq = _c(cu_seqlens_q, np.int32)
        ck = _c(cu_seqlens_k, np.int32)
        kc = _c(k_cache, np.uint16)
        vc = _c(v_cache, np.uint16)
        Tq, Hq, D = q.shape
        NB, BS, Hkv, D2 = kc.shape
        assert D == D2 and Hq % Hkv == 0 and k.shape == (Tq, Hkv, D) and v.shape == k.shape
        B = len(cq) - 1
        bt = None if block_tables is None else _c(block_tables, np.int32)
        out = np.zeros((Tq, Hq, D), dtype=np.float64)
        nt = num_threads or self.max_threads()
        rc = self.lib.oracle_paged_prefill(_ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p),
                                           _ptr(cq, _i32p), _ptr(ck, _i32p), B, _ptr(bt, _i32p),
                                           0 if bt is None else bt.shape[1], _ptr(kc, _u16p),
                                           _ptr(vc, _u16p), NB, BS, Hkv, D, Hq, float(scale),
                                           _ptr(out, _f64p), nt)
        if rc == -2:
            raise ValueError("invalid sequence lengths (k_len < q_len, or prefix without table)")
        if rc:
            raise IndexError("block table walk left the pool")
        return out


    # -- Whole-block moves ----------------------------------------------------------------------
    def copy_blocks(self, k_cache, v_cache, pairs):
        """Return (k_cache', v_cache', skipped) after copying pairs[i,0] -> pairs[i,1]."""
        kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
        vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
        pr = _c(pairs, np.int32)
        bad = self.lib.oracle_copy_blocks(_ptr(kc, _u16p), _ptr(vc, _u16p), kc.shape[0],
                                          int(np.prod(kc.shape[1:])), _ptr(pr, _i32p),
                                          pr.shape[0])
        return kc, vc, int(bad)

    def gather_blocks(self, k_cache, v_cache, ids):
        kc = _c(k_cache, np.uint16)
        vc = _c(v_cache, np.uint16)
        ids = _c(ids, np.int32)
        ok = np.zeros((len(ids),) + kc.shape[1:], np.uint16)
        ov = np.zeros_like(ok)
        bad = self.lib.oracle_gather_blocks(_ptr(kc, _u16p), _ptr(vc, _u16p), kc.shape[0],
                                            int(np.prod(kc.shape[1:])), _ptr(ids, _i32p),
                                            len(ids), _ptr(ok, _u16p), _ptr(ov, _u16p))
        return ok, ov, int(bad)

    def scatter_blocks(self, in_k, in_v, ids, k_cache, v_cache):
        kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
        vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
        ik = _c(in_k, np.uint16)
        iv = _c(in_v, np.uint16)
        ids = _c(ids, np.int32)
        bad = self.lib.oracle_scatter_blocks(_ptr(ik, _u16p), _ptr(iv, _u16p), _ptr(ids, _i32p),
                                             len(ids), _ptr(kc, _u16p), _ptr(vc, _u16p),
                                             kc.shape[0], int(np.prod(kc.shape[1:])))
        return kc, vc, int(bad)


    # -- Chained block hashes -------------------------------------------------------------------
    def xxh64(self, data: bytes, seed: int = 0) -> int:
        return int(self.lib.oracle_xxh64(data, len(data), seed))

    def block_hashes(self, token_ids, cu_seqlens, block_size: int, max_blocks: int):
        """Return ([num_seqs, max_blocks] uint64 with unhashed entries 0, clamped count)."""
        tok = _c(token_ids, np.int32)
        cu = _c(cu_seqlens, np.int32)
        B = len(cu) - 1
        out = np.zeros((B, max_blocks), np.uint64)
        n = self.lib.oracle_block_hashes(_ptr(tok, _i32p), _ptr(cu, _i32p), B, block_size,
                                         max_blocks,
                                         out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
        return out, int(n)


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
