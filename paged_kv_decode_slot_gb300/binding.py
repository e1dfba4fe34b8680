"""ctypes binding of libpagedkv: the C ABI's entry points under the same names.

Argument marshalling only: each function checks dtypes, shapes and devices of
its torch tensors, takes their device pointers and the current CUDA stream,
and calls the library.  Every step of the computation runs in the library's
CUDA kernels.  Functions return the C status code (0 = PKV_OK); ``check``
turns a non-zero status into a ``PkvError``.

The library must be built (``paged_kv_decode_slot_gb300.build``); importing
this module without it raises ImportError -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH as _BUILT_LIB

# PKV_LIBRARY selects another build of the same library (for example one compiled with other
# pipeline depths); by default the in-tree build is loaded.
LIB_PATH = os.environ.get("PKV_LIBRARY") or _BUILT_LIB

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libpagedkv.so is not built ({LIB_PATH}); run __graft_entry__.build()")

_lib = ctypes.CDLL(LIB_PATH)

PKV_OK = 0
PKV_ERR_NULL = -1
PKV_ERR_SHAPE = -2
PKV_ERR_UNSUPPORTED = -3
PKV_ERR_RANGE = -4
PKV_ERR_CUDA = -5
PKV_ERR_ALIGN = -6
PKV_ERR_WORKSPACE = -7

PKV_FLAG_BLOCK_RANGE = 1
PKV_FLAG_SLOT_RANGE = 2
PKV_FLAG_CTX_RANGE = 4
PKV_FLAG_TIMEOUT = 8
PKV_FLAG_OUT_RANGE = 16
PKV_FLAG_GROUP_RANGE = 32

BLOCK_SIZE = 16


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64

_lib.pkv_kv_bytes.argtypes = [_I64] * 5
_lib.pkv_kv_bytes.restype = ctypes.c_uint64
_lib.pkv_slot_mapping.argtypes = [_P, _I32, _P, _I32, _I32, _P, _P, _P]
_lib.pkv_append.argtypes = [_P, _P, _P, _I32, _P, _P, CacheDesc, _P, _P]
_lib.pkv_decode_attn.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P, _P,
                                 CacheDesc, _P, _P]
_lib.pkv_splitk_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
_lib.pkv_splitk_workspace_bytes.restype = ctypes.c_size_t
_lib.pkv_decode_attn_splitk.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P,
                                        _P, CacheDesc, _I32, _I32, _P, ctypes.c_size_t, _P, _P]
_lib.pkv_decode_attn_partitions.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float,
                                            CacheDesc, _I32, _I32, _P, _P, _P, _P]
_lib.pkv_lse_merge.argtypes = [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P]
_lib.pkv_gather.argtypes = [_P, _P, _P, _I32, _P, _P, _I32, _P, _P, _I64, CacheDesc, _P, _P]
_lib.pkv_read_err_flag.argtypes = [_P, _P, _P]
_lib.pkv_status_string.argtypes = [ctypes.c_int]
_lib.pkv_status_string.restype = ctypes.c_char_p
_lib.pkv_last_error.argtypes = []
_lib.pkv_last_error.restype = ctypes.c_char_p


class PkvError(RuntimeError):
    def __init__(self, status: int):
        msg = _lib.pkv_status_string(status).decode()
        if status == PKV_ERR_CUDA:
            msg += ": " + _lib.pkv_last_error().decode()
        super().__init__(f"libpagedkv status {status}: {msg}")
        self.status = status


def check(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status)


def library():
    """The loaded ctypes library (for tests that inspect exports)."""
    return _lib


# ---------------------------------------------------------------------------------------------
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# The pools and the workspaces must be device memory (the pools are read by TMA).  Every other
# argument may also be pinned (page-locked) host memory, which the kernels read and write in place
# (on a GB300 over NVLink-C2C) -- a step's inputs and outputs need no copies then.
_DEVICE_ONLY = ("k_cache", "v_cache", "workspace", "part_out", "part_lse")


def _need(t, dtype, ndim, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda and (name in _DEVICE_ONLY or not t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + ("" if name in _DEVICE_ONLY else " or pinned host memory"))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _opt(t, dtype, ndim, name):
    if t is not None:
        _need(t, dtype, ndim, name)


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    nb, bs, K, H = k_cache.shape
    return CacheDesc(nb, bs, K, H)


# ---------------------------------------------------------------------------------------------
def pkv_kv_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int, bytes_per_elem: int) -> int:
    return int(_lib.pkv_kv_bytes(layers, kv_heads, head_dim, tokens, bytes_per_elem))


def pkv_slot_mapping(block_tables, context_lens, num_blocks: int, slot_mapping, err_flag=None,
                     stream=None) -> int:
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B = context_lens.shape[0]
    if block_tables.shape[0] != B or slot_mapping.shape[0] != B:
        raise ValueError("batch sizes differ")
    return _lib.pkv_slot_mapping(_ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B,
                                 num_blocks, _ptr(slot_mapping), _ptr(err_flag), _stream(stream))


def pkv_append(k_new, v_new, slot_mapping, k_cache, v_cache, err_flag=None, stream=None) -> int:
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, 3, n)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, 4, n)
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    _opt(err_flag, torch.int32, 1, "err_flag")
    T = k_new.shape[0]
    if slot_mapping.shape[0] != T or tuple(k_new.shape[1:]) != tuple(k_cache.shape[2:]):
        raise ValueError("k_new [T, K, H] must match slot_mapping [T] and k_cache [nb, 16, K, H]")
    if v_new.shape != k_new.shape or v_cache.shape != k_cache.shape:
        raise ValueError("K and V shapes differ")
    return _lib.pkv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(k_cache),
                           _ptr(v_cache), cache_desc(k_cache), _ptr(err_flag), _stream(stream))


def _attn_common(q, k_cache, v_cache, block_tables, context_lens):
    _need(q, torch.bfloat16, 3, "q")
    _need(k_cache, torch.bfloat16, 4, "k_cache")
    _need(v_cache, torch.bfloat16, 4, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    if v_cache.shape != k_cache.shape:
        raise ValueError("K and V pools differ in shape")
    B = q.shape[0]
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("batch sizes differ")
    if q.shape[2] != k_cache.shape[3]:
        raise ValueError("head_dim of q and the cache differ")


def pkv_decode_attn(q, k_cache, v_cache, block_tables, context_lens, scale: float, out, lse_out=None,
                    err_flag=None, stream=None) -> int:
    _attn_common(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(err_flag, torch.int32, 1, "err_flag")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    B, N, _ = q.shape
    return _lib.pkv_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                block_tables.shape[1], _ptr(context_lens), B, N, float(scale),
                                _ptr(out), _ptr(lse_out), cache_desc(k_cache), _ptr(err_flag),
                                _stream(stream))


# The partitioned attention entry points merge inside their one launch when the G x max_partitions
# log-sum-exp weights of a unit fit the kernel's drained ring, else in a pkv_lse_merge launch.
IN_KERNEL_MERGE_WEIGHTS = 8192


def split_attention_launches(num_q_heads: int, num_kv_heads: int, max_partitions: int) -> int:
    """Kernel launches of one partitioned attention call (pkv_decode_attn_splitk, pkv_decode_step,
    and the e4m3 forms)."""
    return 1 if (num_q_heads // num_kv_heads) * max_partitions <= IN_KERNEL_MERGE_WEIGHTS else 2


def multi_attention_launches(max_partitions: int, tcgen05: bool) -> int:
    """Kernel launches of one partitioned pkv_decode_attn_multi call: the mma.sync column kernel's
    last CTA of each (sequence, KV head, chunk of 32 rows) merges the chunk when its
    32 x max_partitions weights fit; otherwise, and always after the tcgen05 kernel, a
    pkv_lse_merge launch follows."""
    return 1 if not tcgen05 and 32 * max_partitions <= IN_KERNEL_MERGE_WEIGHTS else 2


def pkv_splitk_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_partitions: int) -> int:
    return int(_lib.pkv_splitk_workspace_bytes(num_seqs, num_q_heads, head_dim, max_partitions))


def max_partitions_for(max_blocks_per_seq: int, partition_blocks: int) -> int:
    return max(1, -(-max_blocks_per_seq // partition_blocks))


def tapered_partitions_for(max_blocks_per_seq: int, partition_blocks: int) -> int:
    """Partitions the tapered layout needs (partition 0 of partition_blocks // 2 blocks, the others
    of partition_blocks): the split entry points taper when max_partitions is at least this and
    num_seqs x num_kv_heads >= the SM count."""
    h = partition_blocks // 2
    if partition_blocks < 2 or max_blocks_per_seq <= h:
        return max_partitions_for(max_blocks_per_seq, partition_blocks)
    return 1 + -(-(max_blocks_per_seq - h) // partition_blocks)


def pkv_decode_attn_splitk(q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                           partition_blocks: int, max_partitions: int, workspace, lse_out=None,
                           err_flag=None, stream=None) -> int:
    _attn_common(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(err_flag, torch.int32, 1, "err_flag")
    _need(workspace, torch.uint8, 1, "workspace")
    B, N, _ = q.shape
    return _lib.pkv_decode_attn_splitk(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       block_tables.shape[1], _ptr(context_lens), B, N, float(scale),
                                       _ptr(out), _ptr(lse_out), cache_desc(k_cache),
                                       partition_blocks, max_partitions, _ptr(workspace),
                                       workspace.numel(), _ptr(err_flag), _stream(stream))


_lib.pkv_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P, _P,
                                 _P, CacheDesc, _I32, _I32, _P, ctypes.c_size_t, _P, _P]


def pkv_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                    lse_out=None, slot_mapping_out=None, partition_blocks: int = 0,
                    max_partitions: int = 0, workspace=None, err_flag=None, stream=None) -> int:
    _attn_common(q, k_cache, v_cache, block_tables, context_lens)
    _need(k_new, torch.bfloat16, 3, "k_new")
    _need(v_new, torch.bfloat16, 3, "v_new")
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(slot_mapping_out, torch.int64, 1, "slot_mapping_out")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, N, _ = q.shape
    if tuple(k_new.shape) != (B, k_cache.shape[2], k_cache.shape[3]) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, K, H]")
    return _lib.pkv_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, N,
                                float(scale), _ptr(out), _ptr(lse_out), _ptr(slot_mapping_out),
                                cache_desc(k_cache), partition_blocks, max_partitions, _ptr(workspace),
                                0 if workspace is None else workspace.numel(), _ptr(err_flag),
                                _stream(stream))


_lib.pkv_quantize_fp8.argtypes = [_P, _I64, _I32, _I32, _P, _I32, _P, _P]
_lib.pkv_append_fp8.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _P, _P, CacheDesc, _P, _P]
_lib.pkv_decode_attn_fp8.argtypes = [_P, _P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P,
                                     _P, CacheDesc, _I32, _I32, _P, ctypes.c_size_t, _P, _P]
_lib.pkv_decode_step_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32,
                                     ctypes.c_float, _P, _P, _P, CacheDesc, _I32, _I32, _P,
                                     ctypes.c_size_t, _P, _P]


def _need_fp8_pool(t, name):
    _need(t, torch.uint8, 4, name)


def scale_block_stride(k_scale, v_scale, num_kv_heads: int) -> int:
    """0 for per-KV-head scales [K]; K for per-(physical block, KV head) scales [num_blocks, K]."""
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 CUDA tensor")
    if k_scale.shape != v_scale.shape:
        raise ValueError("k_scale and v_scale shapes differ")
    if k_scale.dim() == 1 and k_scale.shape[0] == num_kv_heads:
        return 0
    if k_scale.dim() == 2 and k_scale.shape[1] == num_kv_heads:
        return num_kv_heads
    raise ValueError("scales must be [K] (per KV head) or [num_blocks, K] (per block and KV head)")


def pkv_quantize_fp8(src, scale, dst, stream=None) -> int:
    """e4m3 codes of a bf16 tensor [..., K, H] into dst (uint8) with per-KV-head scales [K], or of
    a pool [num_blocks, 16, K, H] with per-(block, head) scales [num_blocks, K]."""
    if src.dtype != torch.bfloat16 or dst.dtype != torch.uint8 or scale.dtype != torch.float32:
        raise TypeError("src bf16, scale float32, dst uint8")
    for t, n in ((src, "src"), (scale, "scale"), (dst, "dst")):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CUDA tensor")
    if src.shape != dst.shape:
        raise ValueError("src and dst shapes differ")
    K, H = src.shape[-2], src.shape[-1]
    stride = scale_block_stride(scale, scale, K)
    if stride and (src.dim() != 4 or src.shape[0] != scale.shape[0]):
        raise ValueError("per-block scales quantize a whole pool [num_blocks, 16, K, H]")
    return _lib.pkv_quantize_fp8(_ptr(src), src.numel() // (K * H), K, H, _ptr(scale), stride, _ptr(dst),
                                 _stream(stream))


def pkv_append_fp8(k_new, v_new, k_scale, v_scale, slot_mapping, k_cache, v_cache, err_flag=None,
                   stream=None) -> int:
    _need(k_new, torch.bfloat16, 3, "k_new")
    _need(v_new, torch.bfloat16, 3, "v_new")
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    _need_fp8_pool(k_cache, "k_cache")
    _need_fp8_pool(v_cache, "v_cache")
    _opt(err_flag, torch.int32, 1, "err_flag")
    stride = scale_block_stride(k_scale, v_scale, k_cache.shape[2])
    return _lib.pkv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_scale), _ptr(v_scale), stride,
                               _ptr(slot_mapping), k_new.shape[0], _ptr(k_cache), _ptr(v_cache),
                               cache_desc(k_cache), _ptr(err_flag), _stream(stream))


def _fp8_common(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens):
    _need(q, torch.bfloat16, 3, "q")
    _need_fp8_pool(k_cache, "k_cache")
    _need_fp8_pool(v_cache, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    if v_cache.shape != k_cache.shape or q.shape[2] != k_cache.shape[3]:
        raise ValueError("pool shapes / head_dim differ")
    return scale_block_stride(k_scale, v_scale, k_cache.shape[2])


def pkv_decode_attn_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale: float,
                        out, lse_out=None, partition_blocks: int = 0, max_partitions: int = 0,
                        workspace=None, err_flag=None, stream=None) -> int:
    stride = _fp8_common(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens)
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, N, _ = q.shape
    return _lib.pkv_decode_attn_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                    stride, _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, N,
                                    float(scale), _ptr(out), _ptr(lse_out), cache_desc(k_cache),
                                    partition_blocks, max_partitions, _ptr(workspace),
                                    0 if workspace is None else workspace.numel(), _ptr(err_flag),
                                    _stream(stream))


def pkv_decode_step_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                        scale: float, out, lse_out=None, slot_mapping_out=None, partition_blocks: int = 0,
                        max_partitions: int = 0, workspace=None, err_flag=None, stream=None) -> int:
    stride = _fp8_common(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens)
    _need(k_new, torch.bfloat16, 3, "k_new")
    _need(v_new, torch.bfloat16, 3, "v_new")
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(slot_mapping_out, torch.int64, 1, "slot_mapping_out")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, N, _ = q.shape
    return _lib.pkv_decode_step_fp8(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scale), _ptr(v_scale), stride, _ptr(block_tables), block_tables.shape[1],
                                    _ptr(context_lens), B, N, float(scale), _ptr(out), _ptr(lse_out),
                                    _ptr(slot_mapping_out), cache_desc(k_cache), partition_blocks,
                                    max_partitions, _ptr(workspace),
                                    0 if workspace is None else workspace.numel(), _ptr(err_flag),
                                    _stream(stream))


def pkv_decode_attn_partitions(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                               partition_blocks: int, part_out, part_lse, err_flag=None,
                               stream=None) -> int:
    _attn_common(q, k_cache, v_cache, block_tables, context_lens)
    _need(part_out, torch.float32, 4, "part_out")
    _need(part_lse, torch.float32, 3, "part_lse")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, N, H = q.shape
    P = part_out.shape[2]
    if tuple(part_out.shape) != (B, N, P, H) or tuple(part_lse.shape) != (B, N, P):
        raise ValueError("part_out must be [B, N, P, H] and part_lse [B, N, P]")
    return _lib.pkv_decode_attn_partitions(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                           block_tables.shape[1], _ptr(context_lens), B, N,
                                           float(scale), cache_desc(k_cache), partition_blocks, P,
                                           _ptr(part_out), _ptr(part_lse), _ptr(err_flag),
                                           _stream(stream))


def pkv_lse_merge(part_out, part_lse, context_lens, partition_blocks: int, out, lse_out=None,
                  stream=None) -> int:
    _need(part_out, torch.float32, 4, "part_out")
    _need(part_lse, torch.float32, 3, "part_lse")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    B, N, P, H = part_out.shape
    return _lib.pkv_lse_merge(_ptr(part_out), _ptr(part_lse), _ptr(context_lens), B, N, H, P,
                              partition_blocks, _ptr(out), _ptr(lse_out), _stream(stream))


# ---------------------------- several new tokens per sequence ----------------------------
_lib.pkv_slot_mapping_multi.argtypes = [_P, _I32, _P, _I32, _I32, _I32, _P, _P, _P]
_lib.pkv_decode_attn_multi.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, ctypes.c_float, _P,
                                       _P, CacheDesc, _I32, _I32, _P, ctypes.c_size_t, _P, _P]
_lib.pkv_multi_uses_tcgen05.argtypes = [_I32, _I32, _I32, _I32]
_lib.pkv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
_lib.pkv_set_wait_limit_ns.restype = ctypes.c_uint64


_lib.pkv_check_wait_expiry.argtypes = [_P, _P]
# Test builds of the library (-DPKV_TEST_HOOKS, loaded through PKV_LIBRARY) also export
# pkv_debug_withhold_tile; the product library does not.
HAS_TEST_HOOKS = hasattr(_lib, "pkv_debug_withhold_tile")
if HAS_TEST_HOOKS:
    _lib.pkv_debug_withhold_tile.argtypes = [ctypes.c_int64]
    _lib.pkv_debug_withhold_tile.restype = ctypes.c_int64


def pkv_debug_withhold_tile(tile: int) -> int:
    """Test builds only: the attention producers skip this tile of every CTA (-1: off); returns
    the previous value.  Raises on the product library, which has no such hook."""
    if not HAS_TEST_HOOKS:
        raise RuntimeError("pkv_debug_withhold_tile exists only in test builds (-DPKV_TEST_HOOKS)")
    return int(_lib.pkv_debug_withhold_tile(int(tile)))


def pkv_check_wait_expiry(err_flag, stream=None) -> int:
    """One bounded wait that cannot complete: sets PKV_FLAG_TIMEOUT after the current limit."""
    _need(err_flag, torch.int32, 1, "err_flag")
    return _lib.pkv_check_wait_expiry(_ptr(err_flag), _stream(stream))


def pkv_set_wait_limit_ns(limit_ns: int) -> int:
    """Limit of every bounded in-kernel wait for later calls (default 2 s); returns the previous."""
    return int(_lib.pkv_set_wait_limit_ns(int(limit_ns)))
_lib.pkv_copy_blocks.argtypes = [_P, _P, _P, _I32, CacheDesc, _I32, _P, _P]
_lib.pkv_prefix_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32, _I32]
_lib.pkv_prefix_workspace_bytes.restype = ctypes.c_size_t
_lib.pkv_decode_attn_prefix.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P, _P,
                                        _I32, _I32, _I32, _P, _P, CacheDesc, _I32, _I32, _P,
                                        ctypes.c_size_t, _P, _P]


def pkv_slot_mapping_multi(block_tables, context_lens, num_blocks: int, slot_mapping, err_flag=None,
                           stream=None) -> int:
    """slot_mapping int64 [B, T]: slots of each sequence's last T logical positions."""
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(slot_mapping, torch.int64, 2, "slot_mapping")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, T = slot_mapping.shape
    return _lib.pkv_slot_mapping_multi(_ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, T,
                                       num_blocks, _ptr(slot_mapping), _ptr(err_flag), _stream(stream))


def pkv_decode_attn_multi(q, k_cache, v_cache, block_tables, context_lens, scale: float, out, lse_out=None,
                          partition_blocks: int = 0, max_partitions: int = 0, workspace=None,
                          err_flag=None, stream=None) -> int:
    """q, out bf16 [B, T, N, H]; lse_out float32 [B, T, N]."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k_cache, torch.bfloat16, 4, "k_cache")
    _need(v_cache, torch.bfloat16, 4, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(out, torch.bfloat16, 4, "out")
    _opt(lse_out, torch.float32, 3, "lse_out")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, T, N, _ = q.shape
    return _lib.pkv_decode_attn_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                      block_tables.shape[1], _ptr(context_lens), B, T, N, float(scale),
                                      _ptr(out), _ptr(lse_out), cache_desc(k_cache), partition_blocks,
                                      max_partitions, _ptr(workspace),
                                      0 if workspace is None else workspace.numel(), _ptr(err_flag),
                                      _stream(stream))


_lib.pkv_decode_step_multi.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, ctypes.c_float, _P,
                                       _P, _P, CacheDesc, _I32, _I32, _P, ctypes.c_size_t, _P, _P]


def pkv_decode_step_multi(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                          lse_out=None, slot_mapping=None, partition_blocks: int = 0, max_partitions: int = 0,
                          workspace=None, err_flag=None, stream=None) -> int:
    """q, out bf16 [B, T, N, H]; k_new, v_new bf16 [B, T, K, H]; lse_out float32 [B, T, N];
    slot_mapping int64 [B, T] (written)."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k_new, torch.bfloat16, 4, "k_new")
    _need(v_new, torch.bfloat16, 4, "v_new")
    _need(k_cache, torch.bfloat16, 4, "k_cache")
    _need(v_cache, torch.bfloat16, 4, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(out, torch.bfloat16, 4, "out")
    _opt(lse_out, torch.float32, 3, "lse_out")
    _opt(slot_mapping, torch.int64, 2, "slot_mapping")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, T, N, _ = q.shape
    if tuple(k_new.shape) != (B, T, k_cache.shape[2], k_cache.shape[3]) or k_new.shape != v_new.shape:
        raise ValueError("k_new / v_new must be [B, T, K, H]")
    return _lib.pkv_decode_step_multi(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, T, N,
                                      float(scale), _ptr(out), _ptr(lse_out), _ptr(slot_mapping),
                                      cache_desc(k_cache), partition_blocks, max_partitions, _ptr(workspace),
                                      0 if workspace is None else workspace.numel(), _ptr(err_flag),
                                      _stream(stream))


def pkv_multi_uses_tcgen05(num_new: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> bool:
    """Whether pkv_decode_attn_multi runs its tcgen05 column kernel for these sizes."""
    return bool(_lib.pkv_multi_uses_tcgen05(num_new, num_q_heads, num_kv_heads, head_dim))


def pkv_copy_blocks(k_cache, v_cache, src_dst, err_flag=None, stream=None) -> int:
    """Copy-on-write: block src_dst[i, 1] of both pools becomes a copy of block src_dst[i, 0]."""
    if k_cache.dtype not in (torch.bfloat16, torch.uint8) or v_cache.dtype != k_cache.dtype:
        raise TypeError("pools must both be bf16 or both uint8 (e4m3)")
    _need(k_cache, k_cache.dtype, 4, "k_cache")
    _need(v_cache, k_cache.dtype, 4, "v_cache")
    _need(src_dst, torch.int32, 2, "src_dst")
    _opt(err_flag, torch.int32, 1, "err_flag")
    if src_dst.shape[1] != 2 or v_cache.shape != k_cache.shape:
        raise ValueError("src_dst must be [n, 2]; pools must have one shape")
    return _lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst), src_dst.shape[0],
                                cache_desc(k_cache), k_cache.element_size(), _ptr(err_flag),
                                _stream(stream))


def pkv_prefix_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_blocks_per_seq: int,
                               max_prefix_blocks: int, partition_blocks: int,
                               prefix_partition_blocks: int = 0) -> int:
    return int(_lib.pkv_prefix_workspace_bytes(num_seqs, num_q_heads, head_dim, max_blocks_per_seq,
                                               max_prefix_blocks, partition_blocks, prefix_partition_blocks))


def pkv_decode_attn_prefix(q, k_cache, v_cache, block_tables, context_lens, scale: float, group_starts,
                           prefix_blocks, max_group_size: int, max_prefix_blocks: int, out, lse_out=None,
                           partition_blocks: int = 16, workspace=None, err_flag=None, stream=None,
                           prefix_partition_blocks: int = 0) -> int:
    """Decode attention with each group's shared leading blocks attended once per KV head."""
    _need(q, torch.bfloat16, 3, "q")
    _need(k_cache, torch.bfloat16, 4, "k_cache")
    _need(v_cache, torch.bfloat16, 4, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(group_starts, torch.int32, 1, "group_starts")
    _need(prefix_blocks, torch.int32, 1, "prefix_blocks")
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    if group_starts.numel() != prefix_blocks.numel() + 1:
        raise ValueError("group_starts needs one more entry than prefix_blocks")
    B, N, _ = q.shape
    return _lib.pkv_decode_attn_prefix(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       block_tables.shape[1], _ptr(context_lens), B, N, float(scale),
                                       _ptr(group_starts), _ptr(prefix_blocks), prefix_blocks.numel(),
                                       max_group_size, max_prefix_blocks, _ptr(out), _ptr(lse_out),
                                       cache_desc(k_cache), partition_blocks, prefix_partition_blocks,
                                       _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                       _ptr(err_flag), _stream(stream))


_lib.pkv_decode_step_prefix.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P, _P,
                                        _I32, _I32, _I32, _P, _P, _P, CacheDesc, _I32, _I32, _P,
                                        ctypes.c_size_t, _P, _P]


def pkv_decode_step_prefix(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale: float,
                           group_starts, prefix_blocks, max_group_size: int, max_prefix_blocks: int, out,
                           lse_out=None, slot_mapping=None, partition_blocks: int = 16, workspace=None,
                           err_flag=None, stream=None, prefix_partition_blocks: int = 0) -> int:
    """Slot mapping + append + shared-prefix decode attention, the append done by the attention
    launch: k_new, v_new bf16 [B, K, H]; slot_mapping int64 [B] (written)."""
    _need(q, torch.bfloat16, 3, "q")
    _need(k_new, torch.bfloat16, 3, "k_new")
    _need(v_new, torch.bfloat16, 3, "v_new")
    _need(k_cache, torch.bfloat16, 4, "k_cache")
    _need(v_cache, torch.bfloat16, 4, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(group_starts, torch.int32, 1, "group_starts")
    _need(prefix_blocks, torch.int32, 1, "prefix_blocks")
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(slot_mapping, torch.int64, 1, "slot_mapping")
    _opt(workspace, torch.uint8, 1, "workspace")
    _opt(err_flag, torch.int32, 1, "err_flag")
    if group_starts.numel() != prefix_blocks.numel() + 1:
        raise ValueError("group_starts needs one more entry than prefix_blocks")
    B, N, _ = q.shape
    if tuple(k_new.shape) != (B, k_cache.shape[2], k_cache.shape[3]) or k_new.shape != v_new.shape:
        raise ValueError("k_new / v_new must be [B, K, H]")
    return _lib.pkv_decode_step_prefix(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, N,
                                       float(scale), _ptr(group_starts), _ptr(prefix_blocks),
                                       prefix_blocks.numel(), max_group_size, max_prefix_blocks, _ptr(out),
                                       _ptr(lse_out), _ptr(slot_mapping), cache_desc(k_cache), partition_blocks,
                                       prefix_partition_blocks, _ptr(workspace),
                                       0 if workspace is None else workspace.numel(), _ptr(err_flag),
                                       _stream(stream))


def pkv_gather(k_cache, v_cache, block_tables, context_lens, cu_seqlens, k_out, v_out, err_flag=None,
               stream=None) -> int:
    _need(k_cache, torch.bfloat16, 4, "k_cache")
    _need(v_cache, torch.bfloat16, 4, "v_cache")
    _need(block_tables, torch.int32, 2, "block_tables")
    _need(context_lens, torch.int32, 1, "context_lens")
    _need(cu_seqlens, torch.int64, 1, "cu_seqlens")
    _need(k_out, torch.bfloat16, 3, "k_out")
    _need(v_out, torch.bfloat16, 3, "v_out")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B = context_lens.shape[0]
    return _lib.pkv_gather(_ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                           _ptr(context_lens), _ptr(cu_seqlens), B, _ptr(k_out), _ptr(v_out),
                           k_out.shape[0], cache_desc(k_cache), _ptr(err_flag), _stream(stream))


def pkv_read_err_flag(err_flag, stream=None) -> tuple[int, int]:
    """(status, flag value): synchronises the stream and reads the device flag."""
    _need(err_flag, torch.int32, 1, "err_flag")
    host = ctypes.c_int32(0)
    st = _lib.pkv_read_err_flag(_ptr(err_flag), ctypes.byref(host), _stream(stream))
    return st, host.value


def pkv_status_string(status: int) -> str:
    return _lib.pkv_status_string(status).decode()


def pkv_last_error() -> str:
    return _lib.pkv_last_error().decode()


# ---------------------------------------------------------------------------------------------
# Split-KV attention without a workspace, for callers that cannot allocate device memory where
# they run attention (graph capture, allocator callbacks, frameworks that own the heap).
STATIC_SCRATCH_BYTES = 8 << 20

_lib.pkv_decode_attn_splitk_noalloc.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, ctypes.c_float,
                                                _P, _P, CacheDesc, _I32, _I32, _P, _P]


def pkv_decode_attn_splitk_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                                   partition_blocks: int, max_partitions: int, lse_out=None,
                                   err_flag=None, stream=None) -> int:
    """pkv_decode_attn_splitk with the partials in the library's static scratch.

    Needs pkv_splitk_workspace_bytes(B, N, H, max_partitions) <= STATIC_SCRATCH_BYTES, else
    returns PKV_ERR_WORKSPACE.  Calls share the scratch: do not overlap them on the GPU.
    """
    _attn_common(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, torch.bfloat16, 3, "out")
    _opt(lse_out, torch.float32, 2, "lse_out")
    _opt(err_flag, torch.int32, 1, "err_flag")
    B, N, _ = q.shape
    return _lib.pkv_decode_attn_splitk_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                               block_tables.shape[1], _ptr(context_lens), B, N,
                                               float(scale), _ptr(out), _ptr(lse_out),
                                               cache_desc(k_cache), partition_blocks, max_partitions,
                                               _ptr(err_flag), _stream(stream))
