"""The C-ABI library on the CPU: it loads, exports every declared symbol, and validates
arguments on the host before any CUDA call (no GPU is touched by these tests)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_slot_gb300.build import build_library
    path = build_library()
    return ctypes.CDLL(path), path


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pkv_append", "pkv_decode_attn", "pkv_decode_attn_splitk", "pkv_lse_merge",
                 "pkv_gather", "pkv_slot_mapping", "pkv_kv_bytes", "pkv_splitk_workspace_bytes",
                 "pkv_decode_attn_partitions", "pkv_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    cdll, path = lib
    for name in declared_functions():
        assert hasattr(cdll, name), f"{name} declared in pkv.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r"\s[TW]\s+(pkv_\w+)$", out.stdout, flags=re.M))
        assert exported == set(declared_functions()), exported ^ set(declared_functions())


class Desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


P = ctypes.c_void_p
FAKE = 0x10000          # an aligned stand-in device address; host validation never dereferences it


def _attn(cdll, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, ctx=FAKE, out=FAKE, B=4, N=8, max_nb=4,
          desc=(64, 16, 2, 64), lse=None):
    f = cdll.pkv_decode_attn
    f.argtypes = [P, P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, P, P,
                  Desc, P, P]
    return f(q, k, v, bt, max_nb, ctx, B, N, 0.125, out, lse, Desc(*desc), None, None)


def test_host_validation_of_decode_attn(lib):
    cdll, _ = lib
    assert _attn(cdll, q=None) == -1
    assert _attn(cdll, out=None) == -1
    assert _attn(cdll, desc=(64, 16, 2, 96)) == -3        # head_dim
    assert _attn(cdll, desc=(64, 8, 2, 64)) == -3         # block size
    assert _attn(cdll, N=6, desc=(64, 16, 4, 64)) == -2    # N % K
    assert _attn(cdll, N=32, desc=(64, 16, 2, 64)) == -3   # G = 16
    assert _attn(cdll, k=FAKE + 8) == -6                  # TMA needs 16-byte alignment
    assert _attn(cdll, B=-1) == -2
    assert _attn(cdll, max_nb=0) == -2
    assert _attn(cdll, B=0) == 0                          # nothing to do, nothing launched


def test_host_validation_of_splitk_and_merge(lib):
    cdll, _ = lib
    f = cdll.pkv_decode_attn_splitk
    f.argtypes = [P, P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, P, P,
                  Desc, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_size_t, P, P]
    cdll.pkv_splitk_workspace_bytes.restype = ctypes.c_size_t
    need = cdll.pkv_splitk_workspace_bytes(4, 8, 64, 2)
    # part_out, then part_lse, then the merge counters, each region 256-byte aligned
    lse_off = 256 * ((4 * 8 * 2 * 64 * 4 + 255) // 256)
    cnt_off = 256 * ((lse_off + 4 * 8 * 2 * 4 + 255) // 256)
    assert need == cnt_off + 4 * 8 * 4
    args = lambda ws, wsb, pb=2, P_=2, B=4: (FAKE, FAKE, FAKE, FAKE, 4, FAKE, B, 8, 0.125, FAKE, None,
                                            Desc(64, 16, 2, 64), pb, P_, ws, wsb, None, None)
    assert f(*args(None, need)) == -7
    assert f(*args(FAKE, need - 1)) == -7
    assert f(*args(FAKE + 16, need)) == -6                # workspace alignment 256
    assert f(*args(FAKE, need, pb=0)) == -2
    assert f(*args(FAKE, need, B=0)) == 0
    g = cdll.pkv_lse_merge
    g.argtypes = [P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, P, P, P]
    assert g(None, FAKE, FAKE, 4, 8, 64, 2, 2, FAKE, None, None) == -1
    assert g(FAKE, FAKE, FAKE, 4, 8, 64, 0, 2, FAKE, None, None) == -2
    assert g(FAKE, FAKE, FAKE, 0, 8, 64, 2, 2, FAKE, None, None) == 0


def test_host_validation_of_cache_ops(lib):
    cdll, _ = lib
    a = cdll.pkv_append
    a.argtypes = [P, P, P, ctypes.c_int32, P, P, Desc, P, P]
    assert a(FAKE, FAKE, None, 4, FAKE, FAKE, Desc(64, 16, 2, 64), None, None) == -1
    assert a(FAKE, FAKE, FAKE, 4, FAKE + 2, FAKE, Desc(64, 16, 2, 64), None, None) == -6
    assert a(FAKE, FAKE, FAKE, 4, FAKE, FAKE, Desc(64, 16, 2, 60), None, None) == -3
    assert a(FAKE, FAKE, FAKE, 0, FAKE, FAKE, Desc(64, 16, 2, 64), None, None) == 0
    s = cdll.pkv_slot_mapping
    s.argtypes = [P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, P, P, P]
    assert s(FAKE, 4, FAKE, 3, 64, None, None, None) == -1
    assert s(FAKE, 0, FAKE, 3, 64, FAKE, None, None) == -2
    assert s(FAKE, 4, FAKE, 0, 64, FAKE, None, None) == 0
    gth = cdll.pkv_gather
    gth.argtypes = [P, P, P, ctypes.c_int32, P, P, ctypes.c_int32, P, P, ctypes.c_int64, Desc, P, P]
    assert gth(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, FAKE, FAKE, -1, Desc(64, 16, 2, 64), None, None) == -2
    assert gth(FAKE, FAKE, FAKE, 4, FAKE, None, 2, FAKE, FAKE, 9, Desc(64, 16, 2, 64), None, None) == -1


def test_status_strings(lib):
    cdll, _ = lib
    cdll.pkv_status_string.restype = ctypes.c_char_p
    for st in range(-7, 1):
        assert cdll.pkv_status_string(st) and cdll.pkv_status_string(st) != b"unknown status"


def test_library_kv_bytes_matches_pages(lib):
    cdll, _ = lib
    f = cdll.pkv_kv_bytes
    f.argtypes = [ctypes.c_int64] * 5
    f.restype = ctypes.c_uint64
    for (L, K, H, S, nbytes), expected, cite in pins.read_kv_bytes_golden():
        assert f(L, K, H, S, nbytes) == expected, cite


def test_attention_plan():
    from paged_kv_decode_slot_gb300.step import plan_attention
    p = plan_attention(64, 8, 512, 152)                                 # 512 units cover 152 SMs,
    assert (p.mode, p.partition_blocks, p.max_partitions) == ("split", 128, 5)   # long tables split,
    p = plan_attention(64, 8, 512, 152, taper=False)                    # one more partition: taper
    assert (p.mode, p.partition_blocks, p.max_partitions) == ("split", 128, 4)
    assert plan_attention(20, 8, 95, 152).mode == "single"
    assert plan_attention(128, 40, 64, 152).mode == "single"
    p = plan_attention(2, 8, 8192, 152)                                 # long context: 256 blocks
    assert p.mode == "split" and p.partition_blocks == 256 and p.max_partitions == 32
    p = plan_attention(16, 8, 464, 152)                                 # 128 units: 128 blocks
    assert p.mode == "split" and p.partition_blocks == 128 and p.max_partitions == 4
    p = plan_attention(1, 40, 64, 152)                                  # at least 8 blocks
    assert p.mode == "split" and p.partition_blocks == 8
    p = plan_attention(64, 8, 512, 152, partition_blocks=64)            # several waves: tapered
    assert p.mode == "split" and p.max_partitions == 9
    p = plan_attention(16, 8, 512, 152, partition_blocks=64)            # one wave: uniform
    assert p.mode == "split" and p.max_partitions == 8


def test_launch_counts():
    """Launches per partitioned call, as the entry points decide them: the one-token split merges
    in its launch while G x max_partitions weights fit in 8192; the mma.sync column kernel while
    32 x max_partitions do; the tcgen05 column kernel always merges in a second launch."""
    import paged_kv_decode_slot_gb300 as pkv
    assert pkv.IN_KERNEL_MERGE_WEIGHTS == 8192
    assert pkv.split_attention_launches(32, 8, 2048) == 1 and pkv.split_attention_launches(32, 8, 2049) == 2
    assert pkv.multi_attention_launches(256, False) == 1 and pkv.multi_attention_launches(257, False) == 2
    assert pkv.multi_attention_launches(4, True) == 2


def test_tapered_partition_count():
    """Partition 0 of half a partition, then whole ones: one more partition than the uniform
    layout needs unless the table ends within the first half partition."""
    import paged_kv_decode_slot_gb300 as pkv
    for pb in (2, 3, 4, 7, 128, 256):
        h = pb // 2
        for nb in range(1, 3 * pb + 3):
            n = pkv.tapered_partitions_for(nb, pb)
            covered = h + (n - 1) * pb             # blocks the n tapered partitions cover
            assert covered >= nb and (n == 1 or h + (n - 2) * pb < nb), (pb, nb, n)
            assert n <= pkv.max_partitions_for(nb, pb) + 1
    assert pkv.tapered_partitions_for(5, 1) == 5   # no taper below two blocks a partition


def test_decode_step_host_validation(lib):
    cdll, _ = lib
    f = cdll.pkv_decode_step
    f.argtypes = [P, P, P, P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                  P, P, P, Desc, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_size_t, P, P]
    args = lambda kn=FAKE, pb=0, P_=0, ws=None, wsb=0, B=4, slot=None: (
        FAKE, kn, FAKE, FAKE, FAKE, FAKE, 4, FAKE, B, 8, 0.125, FAKE, None, slot, Desc(64, 16, 2, 64),
        pb, P_, ws, wsb, None, None)
    assert f(*args(kn=None)) == -1
    assert f(*args(kn=FAKE + 8)) == -6                  # k_new rows move as 16-byte vectors
    assert f(*args(slot=FAKE + 4)) == -6
    assert f(*args(pb=-1)) == -2
    assert f(*args(pb=2, P_=1)) == -2                   # 1 partition of 2 blocks < 4 blocks
    assert f(*args(pb=2, P_=2)) == -7                   # partitions need the workspace
    assert f(*args(B=0)) == 0


def test_decode_step_prefix_host_validation(lib):
    """pkv_decode_step_prefix: the fused step's own arguments are checked on the host (no GPU)."""
    cdll, _ = lib
    f = cdll.pkv_decode_step_prefix
    I = ctypes.c_int32
    f.argtypes = [P, P, P, P, P, P, I, P, I, I, ctypes.c_float, P, P, I, I, I, P, P, P, Desc, I, I, P,
                  ctypes.c_size_t, P, P]
    cdll.pkv_prefix_workspace_bytes.restype = ctypes.c_size_t
    cdll.pkv_prefix_workspace_bytes.argtypes = [I] * 7
    wsb = cdll.pkv_prefix_workspace_bytes(4, 8, 64, 4, 2, 2, 0)
    assert wsb > 0
    args = lambda kn=FAKE, vn=FAKE, slot=None, B=4, groups=1, ws=FAKE, nbytes=wsb: (
        FAKE, kn, vn, FAKE, FAKE, FAKE, 4, FAKE, B, 8, 0.125, FAKE, FAKE, groups, 4, 2, FAKE, None, slot,
        Desc(64, 16, 2, 64), 2, 0, ws, nbytes, None, None)
    assert f(*args(kn=None)) == -1
    assert f(*args(vn=None)) == -1
    assert f(*args(kn=FAKE + 8)) == -6                  # new rows move as 16-byte vectors
    assert f(*args(slot=FAKE + 4)) == -6
    assert f(*args(ws=None)) == -1
    assert f(*args(nbytes=wsb - 1)) == -7
    assert f(*args(groups=-1)) == -2
    assert f(*args(B=0)) == -2                          # a group of 4 in a batch of none
    assert f(*args(B=0, groups=0)) == 0


def test_multi_kernel_choice():
    """pkv_decode_attn_multi runs the tcgen05 column kernel from 17 query rows per CTA at H = 128
    (rows = min(T * G, 32)), the mma.sync one below that and at H = 64; no GPU work."""
    from paged_kv_decode_slot_gb300 import binding as B
    assert B.pkv_multi_uses_tcgen05(8, 32, 8, 128)        # 32 rows
    assert not B.pkv_multi_uses_tcgen05(4, 32, 8, 128)    # 16 rows
    assert B.pkv_multi_uses_tcgen05(5, 32, 8, 128)        # 20 rows
    assert B.pkv_multi_uses_tcgen05(3, 16, 2, 128)        # G = 8: 24 rows
    assert B.pkv_multi_uses_tcgen05(64, 32, 8, 128)       # chunks of 32 rows
    assert not B.pkv_multi_uses_tcgen05(8, 32, 8, 64)     # H = 64
    assert not B.pkv_multi_uses_tcgen05(1, 64, 8, 128)    # one token, G = 8: 8 rows
    assert not B.pkv_multi_uses_tcgen05(0, 32, 8, 128)


def test_noalloc_refuses_before_any_cuda_call(lib):
    """Every refusal of the no-alloc entry point comes from host validation, before the scratch
    lookup or a launch (this machine has no GPU, so any CUDA call would fail instead)."""
    cdll, _ = lib
    f = cdll.pkv_decode_attn_splitk_noalloc
    f.argtypes = [P, P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, P, P,
                  Desc, ctypes.c_int32, ctypes.c_int32, P, P]
    cdll.pkv_last_error.restype = ctypes.c_char_p

    def call(B=1, N=1, max_nb=1, pb=1, parts=4, desc=(64, 16, 1, 64)):
        return f(FAKE, FAKE, FAKE, FAKE, max_nb, FAKE, B, N, 0.125, FAKE, None, Desc(*desc), pb, parts,
                 None, None)
    assert call(parts=13000) == -3                 # more partitions than the separate merge takes
    assert call(max_nb=8, pb=1, parts=4) == -2     # the partitions do not cover the table
    assert call(B=8, N=32, parts=1024, desc=(64, 16, 8, 128)) == -7   # partials beyond the scratch
    assert b"static scratch" in cdll.pkv_last_error()
    assert call(pb=0) == -2


def test_product_library_has_no_test_hook(lib):
    cdll, _ = lib
    assert not hasattr(cdll, "pkv_debug_withhold_tile")


def test_test_build_exports_the_hook(tmp_path):
    """The -DPKV_TEST_HOOKS variant (used by the GPU failure tests) exports the tile-withholding
    hook declared in tests/pkv_test_hooks.h, and nothing else beyond the product's exports."""
    from paged_kv_decode_slot_gb300.build import build_library
    path = build_library(out=str(tmp_path / "libpagedkv_test_hooks.so"), defines=("PKV_TEST_HOOKS",),
                         build_dir=str(tmp_path / "obj"))
    hooks = ctypes.CDLL(path)
    hooks.pkv_debug_withhold_tile.argtypes = [ctypes.c_int64]
    hooks.pkv_debug_withhold_tile.restype = ctypes.c_int64
    assert hooks.pkv_debug_withhold_tile(3) == -1 and hooks.pkv_debug_withhold_tile(-1) == 3
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r"\s[TW]\s+(pkv_\w+)$", out.stdout, flags=re.M))
        assert exported == set(declared_functions()) | {"pkv_debug_withhold_tile"}


def test_prefix_planner_crossover():
    """The cascade is planned from 3,000 shared tokens for groups of more than 16 query rows (the
    measured crossover of the 20-sequence, 160-row batch lies between 2K and 4K tokens), with
    prefix partitions growing with the prefix (16 to 128 blocks)."""
    from paged_kv_decode_slot_gb300.step import plan_prefix_decode
    assert plan_prefix_decode(1000, 160) == 0
    assert plan_prefix_decode(2000, 160) == 0
    assert plan_prefix_decode(4000, 160) == 32
    assert plan_prefix_decode(8000, 160) == 32
    assert plan_prefix_decode(16000, 160) == 64
    assert plan_prefix_decode(32000, 160) == 128
    assert plan_prefix_decode(100000, 160) == 128
    assert plan_prefix_decode(3000, 24) == 32          # 187 shared blocks
    assert plan_prefix_decode(32000, 16) == 0
