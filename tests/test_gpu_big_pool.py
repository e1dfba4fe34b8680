"""Pools larger than 4 GiB, the sequences' blocks at the top of the pool (GPU).

A decode step on a pool whose byte offsets pass 2^32 -- every block of the batch placed among the
last block ids of a 6.5 GB (bf16) or 4.9 GB (e4m3) pool -- exercises the 64-bit addressing of the
slot mapping, the append, the gather and the TMA tensor maps' block dimension.  The page table
makes the result independent of where the blocks sit ("Optimización de la inferencia", "Página
Atención"; CS336 Lecture 10 transcript 01:20:50), so the GPU must reproduce the oracle run on the
compact pool: the pools' bytes and the slots bit for bit (the slots shifted by the blocks below),
attention within the tolerance of the other tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from devutil import assert_close, bf16_dev, bf16_host, i32_dev, out_f64
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

BIG_BF16 = 200_000  # blocks: 200,000 x 16 x 8 x 128 x 2 B = 6.55 GB per pool
BIG_E4M3 = 300_000  # blocks: 300,000 x 16 x 8 x 128 x 1 B = 4.92 GB per pool


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


@pytest.fixture(autouse=True)
def release_pools():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _at_top(compact: torch.Tensor, nbig: int) -> tuple[torch.Tensor, int]:
    """A pool of nbig blocks holding the compact pool in its last blocks (the rest is never read)."""
    base = nbig - compact.shape[0]
    big = torch.empty((nbig,) + tuple(compact.shape[1:]), dtype=compact.dtype, device="cuda")
    big[base:].copy_(compact)
    return big, base


def _shift(tables: np.ndarray, base: int) -> np.ndarray:
    t = tables.astype(np.int64)
    return np.where(t >= 0, t + base, t).astype(np.int32)


def _workload():
    w = gen.make_workload("big_pool", 191, 32, 8, 128, [1, 17, 300, 1000, 4100])
    assert BIG_BF16 * 16 * w.K * w.H * 2 > 2 ** 32 and BIG_E4M3 * 16 * w.K * w.H > 2 ** 32
    return w


@pytest.mark.parametrize("part_blocks", [0, 8])
def test_bf16_step_and_gather_at_the_top_of_a_big_pool(pkv, oracle, part_blocks):
    w = _workload()
    kc, base = _at_top(bf16_dev(w.k_cache), BIG_BF16)
    vc, _ = _at_top(bf16_dev(w.v_cache), BIG_BF16)
    bt = i32_dev(_shift(w.block_tables, base))
    cl = i32_dev(w.context_lens)
    q = bf16_dev(w.q)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
    P, ws = 0, None
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_decode_step(q, bf16_dev(w.k_new), bf16_dev(w.v_new), kc, vc, bt, cl, w.scale, out, lse,
                                  slots, part_blocks, P, ws, err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref_slots = oracle.slot_mapping(w.block_tables, w.context_lens)
    assert np.array_equal(slots.cpu().numpy(), np.where(ref_slots >= 0, ref_slots + 16 * base, ref_slots))
    kh, vh = w.k_cache.copy(), w.v_cache.copy()
    oracle.append(w.k_new, w.v_new, ref_slots, kh, vh)
    assert np.array_equal(bf16_host(kc[base:]), kh) and np.array_equal(bf16_host(vc[base:]), vh)
    ref, _ = oracle.decode(w.q, kh, vh, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, f"big pool, partitions {part_blocks}")
    # the gather reads the same rows through the shifted table
    ko, vo, cu = oracle.gather(kh, vh, w.block_tables, w.context_lens)
    k_out = torch.empty(int(cu[-1]), w.K, w.H, dtype=torch.bfloat16, device="cuda")
    v_out = torch.empty_like(k_out)
    pkv.check(pkv.pkv_gather(kc, vc, bt, cl, torch.from_numpy(cu[:-1].copy()).cuda(), k_out, v_out, err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert np.array_equal(bf16_host(k_out), ko) and np.array_equal(bf16_host(v_out), vo)


@pytest.mark.parametrize("gran", ["head", "block"])
def test_e4m3_step_at_the_top_of_a_big_pool(pkv, oracle, gran):
    from test_gpu_fp8 import Fp8Case, f32_dev, u8_dev
    w = _workload()
    c = Fp8Case(oracle, w, gran)
    kc, base = _at_top(u8_dev(c.kc8), BIG_E4M3)
    vc, _ = _at_top(u8_dev(c.vc8), BIG_E4M3)
    if gran == "block":  # per-(block, KV head) scales follow their blocks to the top
        ks = np.ones((BIG_E4M3, w.K), dtype=np.float32)
        vs = np.ones((BIG_E4M3, w.K), dtype=np.float32)
        ks[base:], vs[base:] = c.ks, c.vs
    else:
        ks, vs = c.ks, c.vs
    bt = i32_dev(_shift(w.block_tables, base))
    q = bf16_dev(w.q)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
    P = pkv.max_partitions_for(w.max_blocks, 8)
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_decode_step_fp8(q, bf16_dev(w.k_new), bf16_dev(w.v_new), kc, vc, f32_dev(ks), f32_dev(vs), bt,
                                      i32_dev(w.context_lens), w.scale, out, lse, slots, 8, P, ws, err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert np.array_equal(kc[base:].cpu().numpy(), c.kc8_app) and np.array_equal(vc[base:].cpu().numpy(), c.vc8_app)
    ref, _ = c.reference(oracle)
    assert_close(out_f64(out), ref, f"big e4m3 pool, {gran} scales")


def test_multi_token_step_at_the_top_of_a_big_pool(pkv, oracle):
    """Eight new tokens (the tcgen05 column kernel, its producers appending) on the big pool."""
    w = _workload()
    T = 8
    q = gen.normal_bf16(192, 1, (w.B, T, w.N, w.H))
    kn = gen.normal_bf16(192, 2, (w.B, T, w.K, w.H))
    vn = gen.normal_bf16(192, 3, (w.B, T, w.K, w.H))
    kc, base = _at_top(bf16_dev(w.k_cache), BIG_BF16)
    vc, _ = _at_top(bf16_dev(w.v_cache), BIG_BF16)
    bt = i32_dev(_shift(w.block_tables, base))
    qd = bf16_dev(q)
    out = torch.empty_like(qd)
    slots = torch.full((w.B, T), -7, dtype=torch.int64, device="cuda")
    P = pkv.max_partitions_for(w.max_blocks, 8)
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B * T, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert pkv.pkv_multi_uses_tcgen05(T, w.N, w.K, w.H)
    pkv.check(pkv.pkv_decode_step_multi(qd, bf16_dev(kn), bf16_dev(vn), kc, vc, bt, i32_dev(w.context_lens), w.scale,
                                        out, None, slots, 8, P, ws, err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref_slots = oracle.slot_mapping_multi(w.block_tables, w.context_lens, T)
    assert np.array_equal(slots.cpu().numpy(), np.where(ref_slots >= 0, ref_slots + 16 * base, ref_slots))
    kh, vh = w.k_cache.copy(), w.v_cache.copy()
    oracle.append(kn.reshape(-1, w.K, w.H), vn.reshape(-1, w.K, w.H), ref_slots.reshape(-1), kh, vh)
    assert np.array_equal(bf16_host(kc[base:]), kh) and np.array_equal(bf16_host(vc[base:]), vh)
    ref, _ = oracle.decode_multi(q, kh, vh, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, "big pool, eight new tokens")
