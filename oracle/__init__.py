"""fp64 CPU oracle for the paged KV-cache path -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of bench.py may import this package.  The CUDA library never loads it,
and it shares no code with the CUDA library.

``build()`` compiles ``pa_oracle.c`` with gcc into ``_build/libpa_oracle.so``
next to this file; the ctypes wrappers below take numpy arrays (bf16 data as
uint16 bit patterns) and return numpy results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpa_oracle.so")
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the oracle with plain gcc (no vectorisation flags), with
    OpenMP when the compiler has it (it only spreads independent output rows
    over threads; without it the same code runs on one thread)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "pa_oracle.h"))):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-I", _HERE, src,
            "-o", tmp, "-lm"]
    if subprocess.run(base + ["-fopenmp"], capture_output=True).returncode != 0:
        subprocess.check_call(base)
    os.replace(tmp, out)
    return out


_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.POINTER(ctypes.c_int64)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_F64 = ctypes.POINTER(ctypes.c_double)


def _declare(lib):
    lib.oracle_set_threads.restype = None
    lib.oracle_set_threads.argtypes = [ctypes.c_int32]
    lib.oracle_max_threads.restype = ctypes.c_int32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_slot.restype = ctypes.c_int64
    lib.oracle_slot.argtypes = [_I32, ctypes.c_int32, ctypes.c_int64]
    lib.oracle_query_start_loc.restype = None
    lib.oracle_query_start_loc.argtypes = [_I32, ctypes.c_int32, _I32]
    lib.oracle_slot_mapping.restype = None
    lib.oracle_slot_mapping.argtypes = [_I32, ctypes.c_int32, _I32, _I32, ctypes.c_int32,
                                        ctypes.c_int32, _I64]
    lib.oracle_reshape_and_cache.restype = None
    lib.oracle_reshape_and_cache.argtypes = [_U16, _U16, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, _U16, _U16, ctypes.c_int32,
                                             ctypes.c_int32, _I64]
    lib.oracle_kv_bytes_per_token.restype = ctypes.c_int64
    lib.oracle_kv_bytes_per_token.argtypes = [ctypes.c_int32] * 4
    lib.oracle_decode.restype = ctypes.c_int
    _U8 = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_reshape_and_cache_fp8.restype = None
    lib.oracle_reshape_and_cache_fp8.argtypes = [_U16, _U16, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, _U8, _U8, ctypes.c_int32,
                                                 ctypes.c_int32, _I64, ctypes.c_float,
                                                 ctypes.c_float]
    lib.oracle_decode_fp8.restype = ctypes.c_int
    lib.oracle_decode_fp8.argtypes = [_F64, _U16, _U8, _U8, _I32, ctypes.c_int32, _I32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                      ctypes.c_double, ctypes.c_double]
    lib.oracle_prefill_varlen_fp8.restype = ctypes.c_int
    lib.oracle_prefill_varlen_fp8.argtypes = [_F64, _U16, _U8, _U8, _I32, _I32, ctypes.c_int32,
                                              _I32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_double, ctypes.c_double, ctypes.c_double]
    lib.oracle_reshape_and_cache_xsplit.restype = None
    lib.oracle_reshape_and_cache_xsplit.argtypes = [_U16, _U16, ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_int32, _U16, _U16, ctypes.c_int32,
                                                    ctypes.c_int32, _I64]
    lib.oracle_decode_xsplit.restype = ctypes.c_int
    lib.oracle_decode_xsplit.argtypes = [_F64, _U16, _U16, _U16, _I32, ctypes.c_int32, _I32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_double]
    lib.oracle_reshape_and_cache_xsplit_fp8.restype = None
    lib.oracle_reshape_and_cache_xsplit_fp8.argtypes = [_U16, _U16, ctypes.c_int32,
                                                        ctypes.c_int32, ctypes.c_int32, _U8, _U8,
                                                        ctypes.c_int32, ctypes.c_int32, _I64,
                                                        ctypes.c_float, ctypes.c_float]
    lib.oracle_decode_xsplit_fp8.restype = ctypes.c_int
    lib.oracle_decode_xsplit_fp8.argtypes = [_F64, _U16, _U8, _U8, _I32, ctypes.c_int32, _I32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                             ctypes.c_double, ctypes.c_double]
    lib.oracle_map_to_kernel_blocks.restype = None
    lib.oracle_map_to_kernel_blocks.argtypes = [_I32, ctypes.c_int32, ctypes.c_int32, _I32]
    lib.oracle_decode.argtypes = [_F64, _U16, _U16, _U16, _I32, ctypes.c_int32, _I32,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_double]
    lib.oracle_prefill_varlen.restype = ctypes.c_int
    lib.oracle_prefill_varlen.argtypes = [_F64, _U16, _U16, _U16, _I32, _I32, ctypes.c_int32,
                                          _I32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_double]
    lib.oracle_online_softmax.restype = None
    lib.oracle_online_softmax.argtypes = [_F64, _F64, ctypes.c_int32, ctypes.c_int32, _I32,
                                          ctypes.c_int32, _F64, _F64, _F64]
    lib.oracle_merge_partitions.restype = None
    lib.oracle_merge_partitions.argtypes = [_F64, _F64, _F64, ctypes.c_int32, ctypes.c_int32,
                                            _F64]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _p(a: np.ndarray, ty):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ty)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype.itemsize == 2 else a
    return a


class Oracle:
    """numpy front end of one loaded oracle library (default: the built one)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def set_threads(self, n: int) -> None:
        """Threads of the decode / prefill loops (1 by default); the results
        are the same for any count."""
        self.lib.oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def slot(self, block_table_row, block_size: int, position: int) -> int:
        row = np.ascontiguousarray(block_table_row, np.int32)
        return int(self.lib.oracle_slot(_p(row, _I32), block_size, position))

    def query_start_loc(self, q_lens) -> np.ndarray:
        ql = np.ascontiguousarray(q_lens, np.int32)
        out = np.zeros(ql.shape[0] + 1, np.int32)
        self.lib.oracle_query_start_loc(_p(ql, _I32), ql.shape[0], _p(out, _I32))
        return out

    def slot_mapping(self, block_tables, query_start_loc, seq_lens, block_size: int) -> np.ndarray:
        bt = np.ascontiguousarray(block_tables, np.int32)
        qsl = np.ascontiguousarray(query_start_loc, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        out = np.full(int(qsl[-1]), -7, np.int64)
        self.lib.oracle_slot_mapping(_p(bt, _I32), bt.shape[1], _p(qsl, _I32), _p(sl, _I32),
                                     sl.shape[0], block_size, _p(out, _I64))
        return out

    def reshape_and_cache(self, key, value, key_cache, value_cache, slot_mapping):
        """Return updated copies of the two caches (inputs are not modified)."""
        k, v = _u16(key), _u16(value)
        kc, vc = _u16(key_cache).copy(), _u16(value_cache).copy()
        sm = np.ascontiguousarray(slot_mapping, np.int64)
        nb, bs, hkv, d = kc.shape
        assert k.shape == (sm.shape[0], hkv, d)
        self.lib.oracle_reshape_and_cache(_p(k, _U16), _p(v, _U16), sm.shape[0], hkv, d,
                                          _p(kc, _U16), _p(vc, _U16), nb, bs, _p(sm, _I64))
        return kc, vc

    def e4m3_decode(self, codes) -> np.ndarray:
        c = np.asarray(codes, dtype=np.uint8)
        return np.array([self.lib.oracle_e4m3_decode(int(x)) for x in c.ravel()]).reshape(c.shape)

    def e4m3_encode(self, values) -> np.ndarray:
        v = np.asarray(values, dtype=np.float32)
        return np.array([self.lib.oracle_e4m3_encode(float(x)) for x in v.ravel()],
                        dtype=np.uint8).reshape(v.shape)

    def reshape_and_cache_fp8(self, key, value, key_cache, value_cache, slot_mapping,
                              k_scale: float, v_scale: float):
        """bf16 key/value bits -> (new e4m3 key cache, new e4m3 value cache)."""
        k, v = _u16(key), _u16(value)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8).copy()
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8).copy()
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        nb, bs, hkv, d = kc.shape
        u8 = ctypes.POINTER(ctypes.c_uint8)
        self.lib.oracle_reshape_and_cache_fp8(_p(k, _U16), _p(v, _U16), sm.shape[0], hkv, d,
                                              _p(kc, u8), _p(vc, u8), nb, bs, _p(sm, _I64),
                                              k_scale, v_scale)
        return kc, vc

    def decode_fp8(self, q, key_cache, value_cache, block_tables, seq_lens, scale,
                   k_scale: float, v_scale: float) -> np.ndarray:
        q = _u16(q)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        S, hq, d = q.shape
        nb, bs, hkv, _ = kc.shape
        out = np.zeros((S, hq, d), dtype=np.float64)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        rc = self.lib.oracle_decode_fp8(_p(out, _F64), _p(q, _U16), _p(kc, u8), _p(vc, u8),
                                        _p(bt, _I32), bt.shape[1], _p(sl, _I32), S, hq, hkv, d, bs,
                                        scale, k_scale, v_scale)
        if rc != 0:
            raise ValueError(f"oracle_decode_fp8 failed ({rc})")
        return out

    def reshape_and_cache_xsplit(self, key, value, key_cache, value_cache, slot_mapping):
        """x-split caches: key [nb, hkv, d / 8, B, 8], value [nb, hkv, d, B] (bf16 bits).
        Returns updated copies (inputs are not modified)."""
        k, v = _u16(key), _u16(value)
        kc, vc = _u16(key_cache).copy(), _u16(value_cache).copy()
        sm = np.ascontiguousarray(slot_mapping, np.int64)
        nb, hkv, dx, bs, x = kc.shape
        d = dx * x
        assert x == 8 and vc.shape == (nb, hkv, d, bs) and k.shape == (sm.shape[0], hkv, d)
        self.lib.oracle_reshape_and_cache_xsplit(_p(k, _U16), _p(v, _U16), sm.shape[0], hkv, d,
                                                 _p(kc, _U16), _p(vc, _U16), nb, bs, _p(sm, _I64))
        return kc, vc

    def decode_xsplit(self, q, key_cache, value_cache, block_tables, seq_lens,
                      scale) -> np.ndarray:
        q, kc, vc = _u16(q), _u16(key_cache), _u16(value_cache)
        bt = np.ascontiguousarray(block_tables, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        s, hq, d = q.shape
        nb, hkv, dx, bs, x = kc.shape
        assert x == 8 and dx * x == d and vc.shape == (nb, hkv, d, bs)
        out = np.zeros((s, hq, d), np.float64)
        rc = self.lib.oracle_decode_xsplit(_p(out, _F64), _p(q, _U16), _p(kc, _U16),
                                           _p(vc, _U16), _p(bt, _I32), bt.shape[1], _p(sl, _I32),
                                           s, hq, hkv, d, bs, float(scale))
        if rc != 0:
            raise ValueError(f"oracle_decode_xsplit rejected its arguments ({rc})")
        return out

    def reshape_and_cache_xsplit_fp8(self, key, value, key_cache, value_cache, slot_mapping,
                                     k_scale: float, v_scale: float):
        """e4m3 x-split caches: key [nb, hkv, d / 16, B, 16], value [nb, hkv, d, B] (bytes).
        Returns updated copies (inputs are not modified)."""
        k, v = _u16(key), _u16(value)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8).copy()
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8).copy()
        sm = np.ascontiguousarray(slot_mapping, np.int64)
        nb, hkv, dx, bs, x = kc.shape
        d = dx * x
        assert x == 16 and vc.shape == (nb, hkv, d, bs) and k.shape == (sm.shape[0], hkv, d)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        self.lib.oracle_reshape_and_cache_xsplit_fp8(_p(k, _U16), _p(v, _U16), sm.shape[0], hkv,
                                                     d, _p(kc, u8), _p(vc, u8), nb, bs,
                                                     _p(sm, _I64), k_scale, v_scale)
        return kc, vc

    def decode_xsplit_fp8(self, q, key_cache, value_cache, block_tables, seq_lens, scale,
                          k_scale: float, v_scale: float) -> np.ndarray:
        q = _u16(q)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
        bt = np.ascontiguousarray(block_tables, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        s, hq, d = q.shape
        nb, hkv, dx, bs, x = kc.shape
        assert x == 16 and dx * x == d and vc.shape == (nb, hkv, d, bs)
        out = np.zeros((s, hq, d), np.float64)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        rc = self.lib.oracle_decode_xsplit_fp8(_p(out, _F64), _p(q, _U16), _p(kc, u8), _p(vc, u8),
                                               _p(bt, _I32), bt.shape[1], _p(sl, _I32), s, hq,
                                               hkv, d, bs, float(scale), float(k_scale),
                                               float(v_scale))
        if rc != 0:
            raise ValueError(f"oracle_decode_xsplit_fp8 rejected its arguments ({rc})")
        return out

    def map_to_kernel_blocks(self, ids, k: int) -> np.ndarray:
        """Manager block ids (any shape; last axis = blocks) -> kernel block ids."""
        a = np.ascontiguousarray(ids, dtype=np.int32)
        out = np.empty(a.shape[:-1] + (a.shape[-1] * k,), dtype=np.int32)
        self.lib.oracle_map_to_kernel_blocks(_p(a, _I32), a.size, k, _p(out, _I32))
        return out

    def kv_bytes_per_token(self, num_layers, num_kv_heads, head_dim, elem_bytes) -> int:
        return int(self.lib.oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim,
                                                      elem_bytes))

    def decode(self, q, key_cache, value_cache, block_tables, seq_lens, scale) -> np.ndarray:
        q, kc, vc = _u16(q), _u16(key_cache), _u16(value_cache)
        bt = np.ascontiguousarray(block_tables, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        s, hq, d = q.shape
        nb, bs, hkv, d2 = kc.shape
        assert d2 == d and bt.shape[0] == s and sl.shape[0] == s
        out = np.zeros((s, hq, d), np.float64)
        rc = self.lib.oracle_decode(_p(out, _F64), _p(q, _U16), _p(kc, _U16), _p(vc, _U16),
                                    _p(bt, _I32), bt.shape[1], _p(sl, _I32), s, hq, hkv, d, bs,
                                    float(scale))
        if rc != 0:
            raise ValueError(f"oracle_decode rejected its arguments ({rc})")
        return out

    def prefill_varlen(self, q, key_cache, value_cache, query_start_loc, seq_lens,
                       block_tables, scale) -> np.ndarray:
        q, kc, vc = _u16(q), _u16(key_cache), _u16(value_cache)
        qsl = np.ascontiguousarray(query_start_loc, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        bt = np.ascontiguousarray(block_tables, np.int32)
        tq, hq, d = q.shape
        nb, bs, hkv, d2 = kc.shape
        assert d2 == d and int(qsl[-1]) <= tq
        out = np.zeros((tq, hq, d), np.float64)
        rc = self.lib.oracle_prefill_varlen(_p(out, _F64), _p(q, _U16), _p(kc, _U16),
                                            _p(vc, _U16), _p(qsl, _I32), _p(sl, _I32),
                                            sl.shape[0], _p(bt, _I32), bt.shape[1], hq, hkv, d,
                                            bs, float(scale))
        if rc != 0:
            raise ValueError(f"oracle_prefill_varlen rejected its arguments ({rc})")
        return out

    def prefill_varlen_fp8(self, q, key_cache, value_cache, query_start_loc, seq_lens,
                           block_tables, scale, k_scale: float, v_scale: float) -> np.ndarray:
        """prefill_varlen over e4m3 caches (uint8 codes) with their scales."""
        q = _u16(q)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
        qsl = np.ascontiguousarray(query_start_loc, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        bt = np.ascontiguousarray(block_tables, np.int32)
        tq, hq, d = q.shape
        nb, bs, hkv, d2 = kc.shape
        assert d2 == d and int(qsl[-1]) <= tq
        out = np.zeros((tq, hq, d), np.float64)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        rc = self.lib.oracle_prefill_varlen_fp8(_p(out, _F64), _p(q, _U16), _p(kc, u8), _p(vc, u8),
                                                _p(qsl, _I32), _p(sl, _I32), sl.shape[0],
                                                _p(bt, _I32), bt.shape[1], hq, hkv, d, bs,
                                                float(scale), float(k_scale), float(v_scale))
        if rc != 0:
            raise ValueError(f"oracle_prefill_varlen_fp8 rejected its arguments ({rc})")
        return out

    def online_softmax(self, s, v, bounds):
        s = np.ascontiguousarray(s, np.float64)
        v = np.ascontiguousarray(v, np.float64)
        b = np.ascontiguousarray(bounds, np.int32)
        out = np.zeros(v.shape[1], np.float64)
        m = ctypes.c_double()
        l = ctypes.c_double()
        self.lib.oracle_online_softmax(_p(s, _F64), _p(v, _F64), s.shape[0], v.shape[1],
                                       _p(b, _I32), b.shape[0] - 1, _p(out, _F64),
                                       ctypes.byref(m), ctypes.byref(l))
        return out, m.value, l.value

    def merge_partitions(self, m_parts, l_parts, o_parts) -> np.ndarray:
        m = np.ascontiguousarray(m_parts, np.float64)
        l = np.ascontiguousarray(l_parts, np.float64)
        o = np.ascontiguousarray(o_parts, np.float64)
        out = np.zeros(o.shape[1], np.float64)
        self.lib.oracle_merge_partitions(_p(m, _F64), _p(l, _F64), _p(o, _F64), m.shape[0],
                                         o.shape[1], _p(out, _F64))
        return out
