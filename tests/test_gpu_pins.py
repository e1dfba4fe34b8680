"""Two special cases of the attention definition, pinned on every GPU path the steps run.

Block permutation.  Where a sequence's blocks sit in the pool does not matter, only the table
that reaches them ("Optimización de la inferencia", "Página Atención": fixed-size pages anywhere
in GPU memory; CS336 Lecture 10 transcript 01:20:50).  Moving every physical block of the pools
(and, for e4m3 pools with per-block scales, its scale row) to another id and rewriting the tables
to match must leave every output bit-identical: the kernels visit logical blocks in the same
order whatever their ids, so only addresses change.  Checked on the default decode step (tapered
partitions, in-kernel merge, fused append), the e4m3 fused step with per-(block, KV head) scales
(two tiles per consumer step and one), several new tokens on the mma.sync (T = 4) and tcgen05
(T = 8) column kernels, and the shared-prefix cascade.

Constant V.  With V = c for every token, softmax weights summing to one give out = c whatever the
logits ("Construye el mismo", Step 2: the normalised weights multiply V).  The bf16 kernels sum
the same rounded weights they multiply V by, so the fp32 ratio differs from c by a few fp32
roundings -- far below half a bf16 step -- and the bf16 output must be exactly c.  So must the
e4m3 output with one scale per KV head when code * scale is a bf16 value; with per-(block, head)
scales the running sum takes unrounded weights and the output is c within 2^-9 relative.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from devutil import appended_host_cache, assert_close, assert_lse_close, bf16_dev, i32_dev, out_f64, upload
from paged_kv_decode_slot_gb300 import inputs as gen
from test_gpu_fp8 import Fp8Case, f32_dev, u8_dev
from test_gpu_multi_prefix import MultiCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _wide_batch(name: str, seed: int, B: int, N: int = 32, K: int = 8) -> gen.Workload:
    """B ragged sequences (1 .. 4000 tokens, one of 2,500) over K KV heads: with B * K at least the
    SM count the planner's plan is the tapered 128-block split with the in-kernel merge."""
    lens = gen.uniform_int(seed, 9, B, 1, 4000)
    lens[B // 2] = 2500
    return gen.make_workload(name, seed, N, K, 128, lens)


def _perm(num_blocks: int, seed: int) -> torch.Tensor:
    return torch.from_numpy(np.random.default_rng(seed).permutation(num_blocks)).cuda()


def _moved(pool: torch.Tensor, perm: torch.Tensor) -> torch.Tensor:
    """Block i of ``pool`` at id perm[i] (scale rows [num_blocks, K] move the same way)."""
    out = torch.empty_like(pool)
    out[perm] = pool
    return out


def _retabled(tables: torch.Tensor, perm: torch.Tensor) -> torch.Tensor:
    t = tables.long()
    return torch.where(t >= 0, perm[t.clamp(min=0)], t).to(torch.int32).contiguous()


def _moved_slots(slots: torch.Tensor, perm: torch.Tensor) -> torch.Tensor:
    return torch.where(slots >= 0, perm[(slots // 16).clamp(min=0)] * 16 + slots % 16, slots)


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return bool(torch.equal(a, b))


# ------------------------------------ block permutation ------------------------------------
def test_permutation_default_decode_step(pkv, oracle):
    from paged_kv_decode_slot_gb300.step import DecodeStep
    w = _wide_batch("perm_step", 401, -(-_sms() // 8) + 4)
    d = upload(w)
    perm = _perm(w.num_blocks, 402)
    steps = []
    for moved in (False, True):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kc = _moved(d["k_cache"], perm) if moved else d["k_cache"].clone()
        vc = _moved(d["v_cache"], perm) if moved else d["v_cache"].clone()
        bt = _retabled(d["block_tables"], perm) if moved else d["block_tables"]
        step = DecodeStep(d["q"], d["k_new"], d["v_new"], kc, vc, bt, d["context_lens"], w.scale, err_flag=err)
        step.run()
        assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
        steps.append(step)
    a, b = steps
    assert a.plan.mode == "split" and a.plan.max_partitions == pkv.tapered_partitions_for(
        w.max_blocks, a.plan.partition_blocks), a.plan.describe()
    assert _same(a.out, b.out) and _same(a.lse, b.lse)
    assert _same(_moved_slots(a.slot_mapping, perm), b.slot_mapping)
    assert _same(_moved(a.k_cache, perm), b.k_cache) and _same(_moved(a.v_cache, perm), b.v_cache)
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(a.out), ref, "permutation, default step")
    assert_lse_close(a.lse.cpu().numpy().astype(np.float64), ref_lse, "permutation, default step")


@pytest.mark.parametrize("B", [6, 24], ids=["two_tiles_per_step", "one_tile_per_step"])
def test_permutation_fp8_step_block_scales(pkv, oracle, B):
    from paged_kv_decode_slot_gb300.step import DecodeStepFp8
    w = _wide_batch(f"perm_fp8_{B}", 403, B)
    c = Fp8Case(oracle, w, "block")
    perm = _perm(w.num_blocks, 404)
    permc = perm.cpu().numpy()
    steps = []
    for moved in (False, True):
        d = c.device(appended=False)
        if moved:
            d["k_cache"], d["v_cache"] = _moved(d["k_cache"], perm), _moved(d["v_cache"], perm)
            d["k_scale"], d["v_scale"] = _moved(d["k_scale"], perm), _moved(d["v_scale"], perm)
            d["block_tables"] = _retabled(d["block_tables"], perm)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        step = DecodeStepFp8(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["k_scale"],
                             d["v_scale"], d["block_tables"], d["context_lens"], w.scale, err_flag=err)
        step.run()
        assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
        steps.append(step)
    a, b = steps
    assert _same(a.out, b.out) and _same(a.lse, b.lse)
    assert _same(_moved_slots(a.slot_mapping, perm), b.slot_mapping)
    assert _same(_moved(a.k_cache, perm), b.k_cache) and _same(_moved(a.v_cache, perm), b.v_cache)
    assert np.array_equal(permc[np.argsort(permc)], np.arange(w.num_blocks))
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(a.out), ref, f"permutation, e4m3 step B={B}")
    assert_lse_close(a.lse.cpu().numpy().astype(np.float64), ref_lse, f"permutation, e4m3 step B={B}")


@pytest.mark.parametrize("T", [4, 8], ids=["mma_sync_T4", "tcgen05_T8"])
def test_permutation_multi_token_step(pkv, oracle, T):
    from paged_kv_decode_slot_gb300.step import MultiTokenStep
    w = _wide_batch(f"perm_multi_{T}", 405 + T, 12)
    c = MultiCase(oracle, w, T, 410 + T)
    assert bool(pkv.pkv_multi_uses_tcgen05(T, w.N, w.K, w.H)) == (T == 8)
    d = upload(w)
    perm = _perm(w.num_blocks, 406)
    steps = []
    for moved in (False, True):
        kc = _moved(d["k_cache"], perm) if moved else d["k_cache"].clone()
        vc = _moved(d["v_cache"], perm) if moved else d["v_cache"].clone()
        bt = _retabled(d["block_tables"], perm) if moved else d["block_tables"]
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        step = MultiTokenStep(bf16_dev(c.q), bf16_dev(c.k_new), bf16_dev(c.v_new), kc, vc, bt, d["context_lens"],
                              w.scale, err_flag=err)
        step.run()
        assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
        steps.append(step)
    a, b = steps
    assert _same(a.out, b.out) and _same(a.lse, b.lse)
    assert _same(_moved_slots(a.slot_mapping, perm), b.slot_mapping)
    assert _same(_moved(a.k_cache, perm), b.k_cache)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(a.out), ref, f"permutation, {T} new tokens")
    assert_lse_close(a.lse.cpu().numpy().astype(np.float64), ref_lse, f"permutation, {T} new tokens")


def test_permutation_shared_prefix_cascade(pkv, oracle):
    from paged_kv_decode_slot_gb300.step import PrefixDecodeStep
    w = gen.make_config("prefix_l3_70b")
    starts, pblocks = w.prefix_groups()
    d = upload(w)
    perm = _perm(w.num_blocks, 407)
    outs = []
    for moved in (False, True):
        kc = _moved(d["k_cache"], perm) if moved else d["k_cache"].clone()
        vc = _moved(d["v_cache"], perm) if moved else d["v_cache"].clone()
        bt = _retabled(d["block_tables"], perm) if moved else d["block_tables"]
        step = PrefixDecodeStep(d["q"], d["k_new"], d["v_new"], kc, vc, bt, d["context_lens"], w.scale,
                                i32_dev(starts), i32_dev(pblocks), w.B, int(pblocks.max()))
        step.run()
        outs.append((step.out, step.lse))
    assert _same(outs[0][0], outs[1][0]) and _same(outs[0][1], outs[1][1])


# ------------------------------------ constant V -------------------------------------------
C_VALUES = [0.30078125, -3.0, 0.0009765625, 37.5]   # bf16 values (0.3 rounded, 2^-10, ...)


def _constant_v(w: gen.Workload, c: float) -> gen.Workload:
    """V = c for every cached and new token (NaN poison left where it was)."""
    import dataclasses
    bits = gen.f32_to_bf16_bits(np.array([c], dtype=np.float32))[0]
    vc = w.v_cache.copy()
    vc[vc != gen.BF16_NAN] = bits
    return dataclasses.replace(w, v_cache=vc, v_new=np.full_like(w.v_new, bits))


def _assert_all_c(out: torch.Tensor, c: float, rows_with_keys, what: str):
    got = out.float().cpu().numpy()[rows_with_keys]
    bad = got != np.float32(c)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements differ from {c}, e.g. {got[bad][:4]}"


@pytest.mark.parametrize("c", C_VALUES)
def test_constant_v_bf16_paths(pkv, oracle, c):
    from paged_kv_decode_slot_gb300.step import DecodeStep, MultiTokenStep
    w = _constant_v(_wide_batch("const_v", 421, -(-_sms() // 8) + 4), c)
    w.context_lens[3] = 0                         # an empty sequence keeps 0 / -inf
    keys = np.asarray(w.context_lens) > 0
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.all(np.abs(ref[keys] / c - 1) <= 1e-13)   # the float64 oracle: c up to its rounding
    d = upload(w)
    step = DecodeStep(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                      d["context_lens"], w.scale)
    step.run()
    _assert_all_c(step.out, c, keys, f"default step ({step.plan.describe()})")
    assert_lse_close(step.lse.cpu().numpy().astype(np.float64), ref_lse, "constant V, default step")
    assert torch.all(step.out[3].float() == 0)
    out = torch.empty_like(d["q"])
    pkv.check(pkv.pkv_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                  w.scale, out))
    _assert_all_c(out, c, keys, "single pass")
    P = pkv.max_partitions_for(w.max_blocks, 3)
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, out, 3, P, ws))
    _assert_all_c(out, c, keys, "3-block partitions")
    for T in (4, 8):                              # mma.sync and tcgen05 column kernels
        mc = MultiCase(oracle, w, T, 430 + T)
        vn = np.full_like(mc.v_new, gen.f32_to_bf16_bits(np.array([c], dtype=np.float32))[0])
        kc2, vc2 = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
        mstep = MultiTokenStep(bf16_dev(mc.q), bf16_dev(mc.k_new), bf16_dev(vn), kc2, vc2, d["block_tables"],
                               d["context_lens"], w.scale)
        mstep.run()
        ctx = np.asarray(w.context_lens)
        visible = (ctx[:, None] - T + np.arange(T)[None, :]) >= 0     # token t sees [0, ctx - T + t]
        got = mstep.out.float().cpu().numpy()
        assert np.all(got[visible] == np.float32(c)), f"{T} new tokens"
        assert np.all(got[~visible] == 0)


@pytest.mark.parametrize("gran", ["head", "block"])
def test_constant_v_e4m3(pkv, oracle, gran):
    """e4m3 V pool of one code (1.75 = 0x3E) with V scales that are powers of two: c = 1.75 * s is a
    bf16 value; per-head scales give exactly c, per-block scales c within 2^-9 relative."""
    from paged_kv_decode_slot_gb300.step import DecodeStepFp8
    for B in (6, 24):
        w = _wide_batch(f"const_v8_{B}", 441, B)
        c8 = Fp8Case(oracle, w, gran)
        code = np.uint8(0x3E)                       # 1.75 in e4m3
        assert oracle.e4m3_decode_table()[code] == 1.75
        nan = (c8.vc8 & 0x7F) == 0x7F
        c8.vc8[~nan] = code
        c8.vc8_app[:] = np.where((c8.vc8_app & 0x7F) == 0x7F, c8.vc8_app, code)
        # V scale 2^-(kvh + 1) per head (the same for every block of that head)
        c8.vs = np.broadcast_to(2.0 ** -(1.0 + np.arange(w.K, dtype=np.float32)), c8.vs.shape).astype(np.float32).copy()
        # the new token's V: exactly 1.75 * scale of its head, so that the append quantizes it to 0x3E
        vnew = np.broadcast_to((1.75 * 2.0 ** -(1.0 + np.arange(w.K)))[None, :, None], w.v_new.shape)
        import dataclasses
        c8.w = w = dataclasses.replace(w, v_new=gen.f32_to_bf16_bits(vnew.astype(np.float32)))
        d = c8.device(appended=False)
        step = DecodeStepFp8(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["k_scale"],
                             d["v_scale"], d["block_tables"], d["context_lens"], w.scale)
        step.run()
        assert torch.equal(d["v_cache"].cpu(), torch.from_numpy(c8.vc8_app))
        want = np.repeat(1.75 * 2.0 ** -(1.0 + np.arange(w.K)), w.N // w.K).astype(np.float32)  # per query head
        got = step.out.float().cpu().numpy()
        if gran == "head":
            assert np.all(got == want[None, :, None]), f"B={B}: {np.abs(got - want[None, :, None]).max()}"
        else:
            assert np.all(np.abs(got / want[None, :, None] - 1) <= 2.0 ** -9), f"B={B}"
        ref, ref_lse = c8.reference(oracle)
        assert np.all(np.abs(ref / want[None, :, None] - 1) <= 1e-13)
        assert_lse_close(step.lse.cpu().numpy().astype(np.float64), ref_lse, f"constant V e4m3 B={B}")
