"""The oracle: plain float64 CPU restatement of paged decode attention.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; the library
``paged_kv_decode_slot_gb300`` never does, and the two share no code.

The C implementation is ``pkv_oracle.c``; this module compiles it with gcc
and exposes numpy-facing wrappers (argument marshalling only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_D = ctypes.c_double


def compile_oracle(source: str = SOURCE, out: str = LIB_PATH, extra_flags=()) -> str:
    """gcc -O2 the oracle into a shared library (plain C11, libm, pthreads)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                           "-I", _HERE, *extra_flags, "-o", tmp, source, "-lm"])
    os.replace(tmp, out)
    return out


def build_oracle(force: bool = False) -> str:
    hdr = os.path.join(_HERE, "pkv_oracle.h")
    newest = max(os.path.getmtime(SOURCE), os.path.getmtime(hdr))
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < newest:
        compile_oracle()
    return LIB_PATH


def _ptr(a: np.ndarray):
    return a.ctypes.data


class Oracle:
    """numpy wrappers over one compiled copy of the oracle library."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = build_oracle()
        lib = ctypes.CDLL(lib_path)
        lib.oracle_kv_bytes.argtypes = [_I64] * 5
        lib.oracle_kv_bytes.restype = ctypes.c_uint64
        lib.oracle_slot_mapping.argtypes = [_P, _I32, _P, _I32, _I32, _P]
        lib.oracle_append.argtypes = [_P, _P, _P, _I32, _P, _P, _I32, _I32]
        lib.oracle_gather.argtypes = [_P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P]
        lib.oracle_decode.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                      _D, _P, _P, ctypes.c_int]
        lib.oracle_decode_partitions.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                                 _I32, _D, _I32, _I32, _P, _P, ctypes.c_int]
        lib.oracle_lse_merge.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _P, _P]
        lib.oracle_slot_mapping_multi.argtypes = [_P, _I32, _P, _I32, _I32, _I32, _P]
        lib.oracle_decode_multi.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                            _I32, _D, _P, _P, ctypes.c_int]
        lib.oracle_copy_blocks.argtypes = [_P, _P, _P, _I32, _I64]
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = _D
        lib.oracle_quantize_fp8.argtypes = [_P, _I64, _I32, _I32, _P, _I32, _I32, _P]
        lib.oracle_append_fp8.argtypes = [_P, _P, _P, _P, _I32, _I32, _P, _I32, _P, _P, _I32, _I32]
        lib.oracle_decode_fp8.argtypes = [_P, _P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                          _I32, _D, _P, _P, ctypes.c_int]
        self.lib = lib

    # -- KV size -------------------------------------------------------------------
    def kv_bytes(self, layers, kv_heads, head_dim, tokens, bytes_per_elem) -> int:
        return int(self.lib.oracle_kv_bytes(layers, kv_heads, head_dim, tokens, bytes_per_elem))

    # -- slot mapping / append / gather --------------------------------------------
    def slot_mapping(self, block_tables, context_lens, bs=16) -> np.ndarray:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty(cl.shape[0], dtype=np.int64)
        self.lib.oracle_slot_mapping(_ptr(bt), bt.shape[1], _ptr(cl), cl.shape[0], bs, _ptr(out))
        return out

    def append(self, k_new, v_new, slots, k_cache, v_cache):
        """Writes into (and returns) k_cache, v_cache, which must be C-contiguous uint16."""
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        kn = np.ascontiguousarray(k_new, dtype=np.uint16)
        vn = np.ascontiguousarray(v_new, dtype=np.uint16)
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        K, H = kn.shape[1], kn.shape[2]
        self.lib.oracle_append(_ptr(kn), _ptr(vn), _ptr(sl), sl.shape[0], _ptr(k_cache),
                               _ptr(v_cache), K, H)
        return k_cache, v_cache

    def gather(self, k_cache, v_cache, block_tables, context_lens, bs=16):
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        cu = np.zeros(cl.shape[0] + 1, dtype=np.int64)
        cu[1:] = np.cumsum(cl.astype(np.int64))
        K, H = k_cache.shape[2], k_cache.shape[3]
        ko = np.empty((int(cu[-1]), K, H), dtype=np.uint16)
        vo = np.empty((int(cu[-1]), K, H), dtype=np.uint16)
        self.lib.oracle_gather(_ptr(np.ascontiguousarray(k_cache)), _ptr(np.ascontiguousarray(v_cache)),
                               _ptr(bt), bt.shape[1], _ptr(cl), _ptr(cu), cl.shape[0], bs, K, H,
                               _ptr(ko), _ptr(vo))
        return ko, vo, cu

    # -- attention -------------------------------------------------------------------
    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, bs=16, threads=0):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
        vc = np.ascontiguousarray(v_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, N, H = q.shape
        K = kc.shape[2]
        assert N % K == 0 and kc.shape[3] == H
        out = np.empty((B, N, H), dtype=np.float64)
        lse = np.empty((B, N), dtype=np.float64)
        self.lib.oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl),
                               B, N, K, H, bs, float(scale), _ptr(out), _ptr(lse), threads)
        return out, lse

    def decode_partitions(self, q, k_cache, v_cache, block_tables, context_lens, scale,
                          partition_tokens, max_parts, bs=16, threads=0):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
        vc = np.ascontiguousarray(v_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, N, H = q.shape
        K = kc.shape[2]
        po = np.empty((B, N, max_parts, H), dtype=np.float64)
        pl = np.empty((B, N, max_parts), dtype=np.float64)
        self.lib.oracle_decode_partitions(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                          _ptr(cl), B, N, K, H, bs, float(scale),
                                          partition_tokens, max_parts, _ptr(po), _ptr(pl), threads)
        return po, pl

    def lse_merge(self, part_out, part_lse):
        po = np.ascontiguousarray(part_out, dtype=np.float64)
        pl = np.ascontiguousarray(part_lse, dtype=np.float64)
        B, N, P, H = po.shape
        out = np.empty((B, N, H), dtype=np.float64)
        lse = np.empty((B, N), dtype=np.float64)
        self.lib.oracle_lse_merge(_ptr(po), _ptr(pl), B, N, H, P, _ptr(out), _ptr(lse))
        return out, lse


    # -- several query tokens per sequence -----------------------------------------------
    def slot_mapping_multi(self, block_tables, context_lens, T, bs=16) -> np.ndarray:
        """Slots [B, T] of the last T logical positions of each sequence (-1 below position 0)."""
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty((cl.shape[0], T), dtype=np.int64)
        self.lib.oracle_slot_mapping_multi(_ptr(bt), bt.shape[1], _ptr(cl), cl.shape[0], T, bs,
                                           _ptr(out))
        return out

    def decode_multi(self, q, k_cache, v_cache, block_tables, context_lens, scale, bs=16, threads=0):
        """q [B, T, N, H] bf16 bits; query token t attends to tokens [0, ctx - T + t]."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
        vc = np.ascontiguousarray(v_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, T, N, H = q.shape
        K = kc.shape[2]
        out = np.empty((B, T, N, H), dtype=np.float64)
        lse = np.empty((B, T, N), dtype=np.float64)
        self.lib.oracle_decode_multi(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl),
                                     B, T, N, K, H, bs, float(scale), _ptr(out), _ptr(lse), threads)
        return out, lse

    # -- copy-on-write -----------------------------------------------------------------
    def copy_blocks(self, k_cache, v_cache, src_dst):
        """In place: block dst of both pools becomes a copy of block src, pair by pair."""
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        assert k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype
        pairs = np.ascontiguousarray(src_dst, dtype=np.int32).reshape(-1, 2)
        block_bytes = k_cache[0].nbytes
        self.lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0],
                                    block_bytes)
        return k_cache, v_cache

    # -- FP8 (e4m3) cache --------------------------------------------------------------
    def e4m3_encode(self, x: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(x)))

    def e4m3_decode_table(self) -> np.ndarray:
        return np.array([self.lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)

    def quantize_fp8(self, src, scale, bs=16) -> np.ndarray:
        """e4m3 codes of a bf16 array [..., K, H] with per-KV-head scales [K], or of a pool
        [num_blocks, bs, K, H] with per-(block, head) scales [num_blocks, K]."""
        x = np.ascontiguousarray(src, dtype=np.uint16)
        sc = np.ascontiguousarray(scale, dtype=np.float32)
        K, H = x.shape[-2], x.shape[-1]
        rows = x.size // (K * H)
        stride = _scale_stride(sc, K)
        if stride:
            assert rows == sc.shape[0] * bs, "per-block scales need the whole pool"
        out = np.empty(x.shape, dtype=np.uint8)
        self.lib.oracle_quantize_fp8(_ptr(x), rows, K, H, _ptr(sc), stride, bs, _ptr(out))
        return out

    def append_fp8(self, k_new, v_new, k_scale, v_scale, slots, k_cache8, v_cache8, bs=16):
        assert k_cache8.flags.c_contiguous and v_cache8.flags.c_contiguous
        kn = np.ascontiguousarray(k_new, dtype=np.uint16)
        vn = np.ascontiguousarray(v_new, dtype=np.uint16)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        K, H = kn.shape[1], kn.shape[2]
        stride = _scale_stride(ks, K)
        assert _scale_stride(vs, K) == stride
        self.lib.oracle_append_fp8(_ptr(kn), _ptr(vn), _ptr(ks), _ptr(vs), stride, bs, _ptr(sl), sl.shape[0],
                                   _ptr(k_cache8), _ptr(v_cache8), K, H)
        return k_cache8, v_cache8

    def decode_fp8(self, q, k_cache8, v_cache8, k_scale, v_scale, block_tables, context_lens, scale,
                   bs=16, threads=0):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(k_cache8, dtype=np.uint8)
        vc = np.ascontiguousarray(v_cache8, dtype=np.uint8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, N, H = q.shape
        K = kc.shape[2]
        stride = _scale_stride(ks, K)
        assert _scale_stride(vs, K) == stride
        out = np.empty((B, N, H), dtype=np.float64)
        lse = np.empty((B, N), dtype=np.float64)
        self.lib.oracle_decode_fp8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), stride, _ptr(bt),
                                   bt.shape[1], _ptr(cl), B, N, K, H, bs, float(scale), _ptr(out),
                                   _ptr(lse), threads)
        return out, lse


def _scale_stride(scale: np.ndarray, K: int) -> int:
    """0 for per-KV-head scales [K]; K for per-(block, head) scales [num_blocks, K]."""
    if scale.ndim == 1:
        assert scale.shape[0] == K
        return 0
    assert scale.ndim == 2 and scale.shape[1] == K
    return K


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
