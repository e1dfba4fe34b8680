"""Seeded synthetic workloads for paged decode attention.

This module only *draws* inputs: context lengths, block permutations, block
tables, and bf16 bit patterns of q, the K/V pools and the new token's K/V.
It holds none of the attention arithmetic; the CUDA library and the float64
oracle both receive its arrays as plain input bytes.

Layouts (all little-endian, bf16 stored as uint16 bit patterns):

* ``q``             [B, N, H]                bf16
* ``k_cache/v_cache`` [num_blocks, bs, K, H] bf16, the state *before* the
  decode step's append: the slot of each sequence's new token (logical
  position ctx-1) and everything after it in its block hold a NaN poison,
  and so does every pool block no table references.
* ``k_new/v_new``   [B, K, H]                bf16, the token appended this step
* ``block_tables``  [B, max_blocks]          int32, tail entries are -1
* ``context_lens``  [B]                      int32, includes the new token

The paged layout (fixed 16-token blocks reached through a per-sequence block
table that maps logical positions to physical blocks anywhere in the pool)
is the one described in "Optimización de la inferencia", section "Página
Atención", and in CS336 Lecture 10, notes section "分页注意力（PagedAttention）".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_gen.c")
_LIB_PATH = os.path.join(_HERE, "libpkvgen.so")

BF16_NAN = np.uint16(0x7FC0)
BLOCK_SIZE = 16

# Stream ids of the counter-based generator (one independent stream each).
_S_CTX, _S_PERM, _S_Q, _S_KPOOL, _S_VPOOL, _S_KNEW, _S_VNEW, _S_SUFFIX = range(8)


def build_gen(force: bool = False) -> str:
    """Compile the generator into ``libpkvgen.so`` next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _gen():
    global _lib
    if _lib is None:
        build_gen()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.pkvgen_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p,
                                           ctypes.c_int]
        lib.pkvgen_uniform_int.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        lib.pkvgen_permutation.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                           ctypes.c_void_p]
        _lib = lib
    return _lib


def normal_bf16(seed: int, stream: int, shape, mult: float = 1.0, offset: int = 0,
                threads: int = 0) -> np.ndarray:
    """bf16 bit patterns of ``mult * N(0,1)`` draws, as a uint16 array of ``shape``."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    rc = _gen().pkvgen_normal_bf16(seed, stream, offset, n, mult, out.ctypes.data, threads)
    assert rc == 0
    return out.reshape(shape)


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    assert _gen().pkvgen_uniform_int(seed, stream, n, lo, hi, out.ctypes.data) == 0
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    assert _gen().pkvgen_permutation(seed, stream, n, out.ctypes.data) == 0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (test and report helper)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even); used to build constant-valued inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    r[nan] = BF16_NAN
    return r


@dataclass
class Workload:
    name: str
    seed: int
    B: int
    N: int
    K: int
    H: int
    scale: float
    context_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray          # int32 [B, max_blocks]
    num_blocks: int
    q: np.ndarray                     # uint16 [B, N, H]
    k_cache: np.ndarray               # uint16 [num_blocks, bs, K, H]  (pre-append)
    v_cache: np.ndarray
    k_new: np.ndarray                 # uint16 [B, K, H]
    v_new: np.ndarray
    partition_blocks: int = 256
    bs: int = BLOCK_SIZE
    unique_tokens: int | None = None  # physical (deduplicated) tokens, when blocks are shared
    notes: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.N // self.K

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode-attention call reads (logical tokens)."""
        return self.total_tokens * self.K * self.H * 2 * 2

    def unique_kv_bytes(self) -> int:
        t = self.unique_tokens if self.unique_tokens is not None else self.total_tokens
        return t * self.K * self.H * 2 * 2

    def prefix_groups(self):
        """(group_starts int32 [G+1], prefix_blocks int32 [G]) of the sequences that share leading
        blocks: one group of the whole batch for the shared-prefix workloads, else None."""
        full = self.notes.get("shared_blocks")
        if full is None:
            return None
        return (np.array([0, self.B], dtype=np.int32), np.array([full], dtype=np.int32))

    def qo_bytes(self) -> int:
        return 2 * self.B * self.N * self.H * 2

    def append_bytes(self) -> int:
        """k_new/v_new read plus the same bytes written into the cache."""
        return 2 * (2 * self.B * self.K * self.H * 2)


def _nblocks(ctx: np.ndarray) -> np.ndarray:
    return (ctx.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE


def _poison_tails(cache: np.ndarray, tables: np.ndarray, ctx: np.ndarray) -> None:
    """NaN every slot at logical position >= ctx-1 of each sequence's last block."""
    for b, c in enumerate(ctx.tolist()):
        if c <= 0:
            continue
        p = c - 1
        blk = tables[b, p // BLOCK_SIZE]
        cache[blk, p % BLOCK_SIZE:] = BF16_NAN


def make_workload(name: str, seed: int, N: int, K: int, H: int, ctx, *, scale: float | None = None,
                  k_mult: float = 1.0, pool_blocks: int | None = None, pool_factor: float = 1.1,
                  partition_blocks: int = 256, max_blocks: int | None = None,
                  threads: int = 0) -> Workload:
    """A batch of independent sequences with context lengths ``ctx``.

    Physical blocks: a pool of ``pool_blocks`` (default ceil(pool_factor * blocks needed))
    is shuffled with a seeded Fisher-Yates permutation, and sequences take
    consecutive entries of the shuffled order (sequence 0 first).  Pool blocks
    no table references are NaN-poisoned.
    """
    ctx = np.asarray(ctx, dtype=np.int32)
    B = int(ctx.shape[0])
    nb = _nblocks(ctx)
    need = int(nb.sum())
    if pool_blocks is None:
        pool_blocks = max(1, int(math.ceil(pool_factor * need)))
    assert pool_blocks >= need
    mb = int(nb.max()) if max_blocks is None else max_blocks
    mb = max(mb, 1)
    perm = permutation(seed, _S_PERM, pool_blocks)
    tables = np.full((B, mb), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        tables[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += int(nb[b])
    q = normal_bf16(seed, _S_Q, (B, N, H), threads=threads)
    kc = normal_bf16(seed, _S_KPOOL, (pool_blocks, BLOCK_SIZE, K, H), mult=k_mult, threads=threads)
    vc = normal_bf16(seed, _S_VPOOL, (pool_blocks, BLOCK_SIZE, K, H), threads=threads)
    kn = normal_bf16(seed, _S_KNEW, (B, K, H), mult=k_mult, threads=threads)
    vn = normal_bf16(seed, _S_VNEW, (B, K, H), threads=threads)
    used = np.zeros(pool_blocks, dtype=bool)
    used[perm[:need]] = True
    kc[~used] = BF16_NAN
    vc[~used] = BF16_NAN
    _poison_tails(kc, tables, ctx)
    _poison_tails(vc, tables, ctx)
    if scale is None:
        scale = 1.0 / math.sqrt(H)
    return Workload(name=name, seed=seed, B=B, N=N, K=K, H=H, scale=scale, context_lens=ctx,
                    block_tables=tables, num_blocks=pool_blocks, q=q, k_cache=kc, v_cache=vc,
                    k_new=kn, v_new=vn, partition_blocks=partition_blocks)


def make_prefix_workload(name: str, seed: int, N: int, K: int, H: int, B: int, prefix: int,
                         suffix_lo: int, suffix_hi: int, *, pool_factor: float = 1.1,
                         threads: int = 0) -> Workload:
    """Sequences sharing one prompt prefix, stored once, with copy-on-write of its last block.

    The prefix's full blocks are physically shared by every table.  Its last,
    partially filled block is copied (bit for bit) into one private block per
    sequence when that sequence writes its first own token; each sequence's
    suffix then continues in the copy and in further private blocks.  This is
    the sharing with copy-on-write that "Optimización de la inferencia"
    ("Página Atención") and CS336 Lecture 10 (notes, "分页注意力"; transcript
    01:21:58-01:23:17, "if they sample different tokens, you split the block")
    describe.
    """
    bs = BLOCK_SIZE
    full = prefix // bs                   # shared full blocks
    rem = prefix - full * bs              # prefix tokens in the partial block
    assert rem > 0, "this builder models a partially filled last prefix block"
    suffix = uniform_int(seed, _S_SUFFIX, B, suffix_lo, suffix_hi).astype(np.int64)
    ctx = (prefix + suffix).astype(np.int32)
    nb = _nblocks(ctx)
    private = nb - full                   # the CoW copy plus later private blocks
    need = full + 1 + int(private.sum())  # +1: the original partial prefix block stays in the pool
    pool_blocks = int(math.ceil(pool_factor * need))
    perm = permutation(seed, _S_PERM, pool_blocks)
    shared = perm[:full]
    orig_partial = int(perm[full])
    tables = np.full((B, int(nb.max())), -1, dtype=np.int32)
    pos = full + 1
    for b in range(B):
        tables[b, :full] = shared
        tables[b, full:nb[b]] = perm[pos:pos + private[b]]
        pos += int(private[b])
    q = normal_bf16(seed, _S_Q, (B, N, H), threads=threads)
    kc = normal_bf16(seed, _S_KPOOL, (pool_blocks, bs, K, H), threads=threads)
    vc = normal_bf16(seed, _S_VPOOL, (pool_blocks, bs, K, H), threads=threads)
    kn = normal_bf16(seed, _S_KNEW, (B, K, H), threads=threads)
    vn = normal_bf16(seed, _S_VNEW, (B, K, H), threads=threads)
    for b in range(B):                    # copy-on-write of the partial prefix block
        dst = tables[b, full]
        kc[dst, :rem] = kc[orig_partial, :rem]
        vc[dst, :rem] = vc[orig_partial, :rem]
    kc[orig_partial, rem:] = BF16_NAN
    vc[orig_partial, rem:] = BF16_NAN
    used = np.zeros(pool_blocks, dtype=bool)
    used[perm[:need]] = True
    kc[~used] = BF16_NAN
    vc[~used] = BF16_NAN
    _poison_tails(kc, tables, ctx)
    _poison_tails(vc, tables, ctx)
    unique = full * bs + int((ctx.astype(np.int64) - full * bs).sum())
    return Workload(name=name, seed=seed, B=B, N=N, K=K, H=H, scale=1.0 / math.sqrt(H),
                    context_lens=ctx, block_tables=tables, num_blocks=pool_blocks, q=q,
                    k_cache=kc, v_cache=vc, k_new=kn, v_new=vn, unique_tokens=unique,
                    notes={"prefix": prefix, "shared_blocks": full, "orig_partial_block": orig_partial})


# --------------------------------------------------------------------------------------
# The named workloads.  Shapes follow the model shapes the pages discuss: Llama-3-8B
# (32 query / 8 KV heads, head_dim 128), Llama-2-13B MHA (40/40, S = 1024) from CS336
# Lecture 10's worked example, and Llama-3-70B's head shape (64 / 8).
# --------------------------------------------------------------------------------------

CONFIG_NAMES = ("tiny", "l3_8b_b64", "l3_8b_b16", "l2_13b_mha_b1", "l2_13b_mha_b8", "l2_13b_mha_b64",
                "l2_13b_mha_b128", "prefix_l3_70b", "prefix_long_l3_70b", "long_splitk")


def make_config(name: str, threads: int = 0) -> Workload:
    if name == "tiny":
        # 4 sequences, 8 query / 2 KV heads, head_dim 64, a 64-block pool in seeded order.
        return make_workload("tiny", 1, 8, 2, 64, [1, 17, 64, 200], scale=1.0 / 8.0,
                             pool_blocks=64, threads=threads)
    if name == "l3_8b_b64":
        ctx = uniform_int(2, _S_CTX, 64, 512, 8192)
        return make_workload("l3_8b_b64", 2, 32, 8, 128, ctx, threads=threads)
    if name == "l3_8b_b16":
        # A quarter of l3_8b_b64 (its first 16 context lengths; K/V still larger than L2),
        # small enough for full profiler captures.
        ctx = uniform_int(2, _S_CTX, 16, 512, 8192)
        return make_workload("l3_8b_b16", 2, 32, 8, 128, ctx, threads=threads)
    if name.startswith("l3_8b_b") and name[len("l3_8b_b"):].isdigit():
        # Any batch size of the same draw (the first B context lengths of the stream above; B = 64
        # and 16 are the two named workloads), for throughput-versus-batch measurements.
        B = int(name[len("l3_8b_b"):])
        ctx = uniform_int(2, _S_CTX, B, 512, 8192)
        return make_workload(name, 2, 32, 8, 128, ctx, threads=threads)
    if name.startswith("l2_13b_mha_b"):
        B = int(name[len("l2_13b_mha_b"):])
        assert B in (1, 8, 64, 128)
        return make_workload(name, 3, 40, 40, 128, [1024] * B, threads=threads)
    if name == "prefix_l3_70b":
        return make_prefix_workload("prefix_l3_70b", 4, 64, 8, 128, 20, 1000, 16, 512,
                                    threads=threads)
    if name == "prefix_long_l3_70b" or name.startswith("prefix_l3_70b_p"):
        # The same batch with a longer shared prompt: 32,008 tokens (2,000 full shared blocks, 128 MB
        # of K/V per layer, about the GB300's L2) for the named workload, any length for
        # "prefix_l3_70b_p<tokens>" (a partly filled last prefix block: tokens % 16 != 0).
        prefix = 32008 if name == "prefix_long_l3_70b" else int(name[len("prefix_l3_70b_p"):])
        return make_prefix_workload(name, 4, 64, 8, 128, 20, prefix, 16, 512, threads=threads)
    if name == "long_splitk":
        return make_workload("long_splitk", 5, 32, 8, 128, [131072, 32768], k_mult=0.5,
                             partition_blocks=256, threads=threads)
    raise KeyError(name)
