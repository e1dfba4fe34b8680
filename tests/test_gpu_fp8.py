"""FP8 (e4m3) KV cache on the GPU against the oracle.

Quantization and append are byte work: the codes must equal the oracle's bit for bit (NaN
inputs must give a NaN code; its sign bit is not compared).  Attention over e4m3 pools is
compared with the oracle's float64 attention over the dequantized pools, at the bf16 path's
tolerance; the fused fp8 step must equal the separate fp8 calls bit for bit.  Both scale
granularities run: one scale per KV head ([K]) and one per (physical block, KV head)
([num_blocks, K]).
"""
from __future__ import annotations

import dataclasses
import warnings

import numpy as np
import pytest
import torch

from devutil import assert_close, assert_lse_close, bf16_dev, i32_dev, out_f64
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def head_scales(cache_bits: np.ndarray, spread: bool = True) -> np.ndarray:
    """Per-KV-head scale = amax / 448 over the finite values, times (1 + kvh) when ``spread``
    so that a kernel that indexes the wrong head's scale is visibly wrong."""
    rows = cache_bits.reshape(-1, cache_bits.shape[-2], cache_bits.shape[-1])
    x = gen.bf16_bits_to_f32(rows[:: max(1, rows.shape[0] // 4096)])
    amax = np.nanmax(np.abs(np.where(np.isfinite(x), x, np.nan)), axis=(0, 2))
    amax = np.where(np.isfinite(amax) & (amax > 0), amax, 1.0)
    mult = 1.0 + np.arange(amax.shape[0]) if spread else 1.0
    return (amax / 448.0 * mult).astype(np.float32)


def block_scales(cache_bits: np.ndarray) -> np.ndarray:
    """Per-(block, KV head) scale = that block's amax / 448 over its finite values (1 where it has
    none), times (1 + kvh) so that a wrong head's scale is visibly wrong; blocks differ by their
    own maxima, so a wrong block's scale is too."""
    x = gen.bf16_bits_to_f32(cache_bits)                                   # [nb, 16, K, H]
    with np.errstate(invalid="ignore"), warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)                     # all-poison blocks
        amax = np.nanmax(np.abs(np.where(np.isfinite(x), x, np.nan)), axis=(1, 3))  # [nb, K]
    amax = np.where(np.isfinite(amax) & (amax > 0), amax, 1.0)
    return (amax / 448.0 * (1.0 + np.arange(amax.shape[1]))[None, :]).astype(np.float32)


GRANULARITIES = ["head", "block"]


def codes_equal(got: np.ndarray, ref: np.ndarray) -> bool:
    nan_ref = (ref & 0x7F) == 0x7F
    nan_got = (got & 0x7F) == 0x7F
    return bool(np.array_equal(nan_ref, nan_got) and np.array_equal(got[~nan_ref], ref[~nan_ref]))


def u8_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def f32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


class Fp8Case:
    """A workload with its e4m3 pools (oracle-quantized) before and after the append, with one
    scale per KV head or one per (physical block, KV head)."""

    def __init__(self, oracle, w: gen.Workload, granularity: str = "head"):
        self.w = w
        scales = block_scales if granularity == "block" else head_scales
        self.ks = scales(w.k_cache)
        self.vs = scales(w.v_cache)
        self.kc8 = oracle.quantize_fp8(w.k_cache, self.ks)
        self.vc8 = oracle.quantize_fp8(w.v_cache, self.vs)
        self.slots = oracle.slot_mapping(w.block_tables, w.context_lens)
        self.kc8_app, self.vc8_app = self.kc8.copy(), self.vc8.copy()
        oracle.append_fp8(w.k_new, w.v_new, self.ks, self.vs, self.slots, self.kc8_app, self.vc8_app)

    def device(self, appended: bool):
        w = self.w
        return dict(q=bf16_dev(w.q), k_new=bf16_dev(w.k_new), v_new=bf16_dev(w.v_new),
                    k_cache=u8_dev(self.kc8_app if appended else self.kc8),
                    v_cache=u8_dev(self.vc8_app if appended else self.vc8),
                    k_scale=f32_dev(self.ks), v_scale=f32_dev(self.vs),
                    block_tables=i32_dev(w.block_tables), context_lens=i32_dev(w.context_lens))

    def reference(self, oracle):
        w = self.w
        return oracle.decode_fp8(w.q, self.kc8_app, self.vc8_app, self.ks, self.vs, w.block_tables,
                                 w.context_lens, w.scale)


def _attn(pkv, c: Fp8Case, d, part_blocks, err=None):
    w = c.w
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    P, ws = 0, None
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    pkv.check(pkv.pkv_decode_attn_fp8(d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                                      d["block_tables"], d["context_lens"], w.scale, out, lse,
                                      part_blocks, P, ws, err))
    return out, lse


def _step(pkv, c: Fp8Case, d, part_blocks, err=None):
    w = c.w
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
    P, ws = 0, None
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    pkv.check(pkv.pkv_decode_step_fp8(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                      d["k_scale"], d["v_scale"], d["block_tables"], d["context_lens"],
                                      w.scale, out, lse, slots, part_blocks, P, ws, err))
    return out, lse, slots


def test_quantize_matches_oracle_codes(pkv, oracle):
    """Every bf16 value class: normals over a wide range, subnormal results, saturation, ties."""
    rng_rows = 300
    src = gen.normal_bf16(71, 0, (rng_rows, 4, 128), mult=30.0)
    bits = src.copy()
    # a few exact e4m3 midpoints (ties) and values past the saturation bound
    tie_vals = np.array([0.0078125 * 1.5, 1.0625, 1.1875, 17.0, 464.0, 500.0, -464.0, 1e-4, -3e-3],
                        dtype=np.float32)
    bits[0, 0, :tie_vals.size] = gen.f32_to_bf16_bits(tie_vals)
    scale = np.array([1.0, 0.5, 0.03125, 3.0], dtype=np.float32)
    ref = oracle.quantize_fp8(bits, scale)
    dst = torch.empty(bits.shape, dtype=torch.uint8, device="cuda")
    pkv.check(pkv.pkv_quantize_fp8(bf16_dev(bits), f32_dev(scale), dst))
    got = dst.cpu().numpy()
    assert codes_equal(got, ref), f"{int(np.sum(got != ref))} codes differ"


def test_quantize_block_scales_matches_oracle(pkv, oracle):
    """A whole pool quantized with per-(block, head) scales: codes equal the oracle's."""
    w = gen.make_workload("p8_qblk", 86, 16, 4, 128, [33, 170, 300, 9])
    for cache in (w.k_cache, w.v_cache):
        sc = block_scales(cache)
        ref = oracle.quantize_fp8(cache, sc)
        dst = torch.empty(cache.shape, dtype=torch.uint8, device="cuda")
        pkv.check(pkv.pkv_quantize_fp8(bf16_dev(cache), f32_dev(sc), dst))
        assert codes_equal(dst.cpu().numpy(), ref)


def test_quantize_every_bf16_bit_pattern(pkv, oracle):
    """All 65536 bf16 patterns (NaNs and infinities included) at two scales."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 1, 128)
    for s in (1.0, 0.0625):
        scale = np.array([s], dtype=np.float32)
        ref = oracle.quantize_fp8(bits, scale)
        dst = torch.empty(bits.shape, dtype=torch.uint8, device="cuda")
        pkv.check(pkv.pkv_quantize_fp8(bf16_dev(bits), f32_dev(scale), dst))
        assert codes_equal(dst.cpu().numpy(), ref), f"scale {s}"


CASES = [
    ("tiny", lambda: gen.make_workload("p8_tiny", 81, 8, 2, 128, [1, 7, 16, 17, 40])),
    ("ragged_gqa4", lambda: gen.make_workload("p8_ragged", 82, 32, 8, 128,
                                              gen.uniform_int(82, 9, 12, 1, 1500))),
    ("mha", lambda: gen.make_workload("p8_mha", 83, 8, 8, 128, [1, 16, 17, 200, 333])),
    ("gqa8", lambda: gen.make_workload("p8_gqa8", 84, 16, 2, 128, [31, 32, 33, 700])),
]


@pytest.mark.parametrize("gran", GRANULARITIES)
def test_append_fp8_matches_oracle(pkv, oracle, gran):
    c = Fp8Case(oracle, CASES[1][1](), gran)
    d = c.device(appended=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_append_fp8(d["k_new"], d["v_new"], d["k_scale"], d["v_scale"],
                                 torch.from_numpy(c.slots).cuda(), d["k_cache"], d["v_cache"], err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert codes_equal(d["k_cache"].cpu().numpy(), c.kc8_app)
    assert codes_equal(d["v_cache"].cpu().numpy(), c.vc8_app)


@pytest.mark.parametrize("gran", GRANULARITIES)
@pytest.mark.parametrize("part_blocks", [0, 2, 7])
@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_decode_attn_fp8_matches_oracle(pkv, oracle, name, make, part_blocks, gran):
    c = Fp8Case(oracle, make(), gran)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _attn(pkv, c, c.device(appended=True), part_blocks, err)
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(out), ref, f"fp8 {name} pb={part_blocks} {gran}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"fp8 {name} pb={part_blocks} {gran}")


@pytest.mark.parametrize("gran", GRANULARITIES)
@pytest.mark.parametrize("part_blocks", [0, 3])
@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_decode_step_fp8_equals_separate_calls(pkv, oracle, name, make, part_blocks, gran):
    c = Fp8Case(oracle, make(), gran)
    # separate: append then attention
    d1 = c.device(appended=False)
    slots1 = torch.empty(c.w.B, dtype=torch.int64, device="cuda")
    pkv.check(pkv.pkv_slot_mapping(d1["block_tables"], d1["context_lens"], c.w.num_blocks, slots1))
    pkv.check(pkv.pkv_append_fp8(d1["k_new"], d1["v_new"], d1["k_scale"], d1["v_scale"], slots1,
                                 d1["k_cache"], d1["v_cache"]))
    out1, lse1 = _attn(pkv, c, d1, part_blocks)
    # fused
    d2 = c.device(appended=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2, lse2, slots2 = _step(pkv, c, d2, part_blocks, err)
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    assert torch.equal(slots1, slots2)
    assert torch.equal(d1["k_cache"], d2["k_cache"]) and torch.equal(d1["v_cache"], d2["v_cache"])
    assert codes_equal(d2["k_cache"].cpu().numpy(), c.kc8_app)
    assert codes_equal(d2["v_cache"].cpu().numpy(), c.vc8_app)
    ref, _ = c.reference(oracle)
    assert_close(out_f64(out2), ref, f"fp8 step {name} pb={part_blocks}")


@pytest.mark.parametrize("gran", GRANULARITIES)
@pytest.mark.parametrize("G", [1, 4, 8])
def test_fp8_every_tail(pkv, oracle, G, gran):
    """Context lengths 1..49 (every in-block position of the new token) for group sizes 1/4/8."""
    c = Fp8Case(oracle, gen.make_workload(f"p8_tail{G}", 90 + G, 2 * G, 2, 128, list(range(1, 50))), gran)
    out, lse = _attn(pkv, c, c.device(appended=True), 0)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(out), ref, f"fp8 tails G={G}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"fp8 tails G={G}")
    out2, lse2, _ = _step(pkv, c, c.device(appended=False), 0)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)


def test_fp8_empty_sequence_and_bad_block(pkv, oracle):
    c = Fp8Case(oracle, gen.make_workload("p8_edge", 95, 8, 2, 128, [0, 20, 33]))
    d = c.device(appended=True)
    bt = d["block_tables"].clone()
    bt[2, 1] = c.w.num_blocks + 3
    d["block_tables"] = bt
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _attn(pkv, c, d, 0, err)
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_BLOCK_RANGE
    assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))
    ref, _ = c.reference(oracle)
    assert_close(out_f64(out[1:2]), ref[1:2], "fp8 edge: the valid sequence")


def test_fp8_full_size_single_and_split(pkv, oracle):
    """Llama-3-8B-shaped batch of 64 (32 query heads, 8 KV heads, 128 dims): the single pass and
    the planner's split, every sequence."""
    w = gen.make_config("l3_8b_b64")
    c = Fp8Case(oracle, w)
    d = c.device(appended=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    from paged_kv_decode_slot_gb300.step import plan_attention
    plan = plan_attention(w.B, w.K, w.max_blocks, sms, mode="split")
    out, lse, _ = _step(pkv, c, d, 0)
    out_s, _ = _attn(pkv, c, d, plan.partition_blocks)
    ref, _ = c.reference(oracle)
    assert_close(out_f64(out), ref, "fp8 l3_8b_b64 single")
    assert_close(out_f64(out_s), ref, "fp8 l3_8b_b64 split")


@pytest.mark.parametrize("name,gran", [("l3_8b_b64", "head"), ("l2_13b_mha_b128", "head"),
                                       ("long_splitk", "head"), ("l3_8b_b16", "head"),
                                       ("l3_8b_b64", "block"), ("l3_8b_b16", "block")])
def test_fp8_step_full_size_in_bench_plan(pkv, oracle, name, gran):
    """The e4m3 decode step as the benchmark times it (DecodeStepFp8 with the planner's plan: one
    tile per step on wide grids, two on grids with fewer units than SMs), every sequence."""
    from paged_kv_decode_slot_gb300.step import DecodeStepFp8
    w = gen.make_config(name)
    c = Fp8Case(oracle, w, gran)
    d = c.device(appended=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = DecodeStepFp8(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["k_scale"],
                         d["v_scale"], d["block_tables"], d["context_lens"], w.scale, err_flag=err)
    step.run()
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert codes_equal(d["k_cache"].cpu().numpy(), c.kc8_app)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(step.out), ref, f"fp8 {name} ({step.plan.describe()})")
    assert_lse_close(step.lse.cpu().numpy().astype(np.float64), ref_lse, f"fp8 {name}")


# ------------------------- per-block scales over a wide range -------------------------------
def wide_scale_workload(B: int) -> gen.Workload:
    """Sequences whose logical blocks hold K and V values of very different magnitudes, so that
    the per-(block, KV head) e4m3 scales of one sequence span four decades (1e-4 .. 1 for V).
    Three kinds of sequence, by b mod 3:
      0  a tiny V scale in the first block, then scales up to 1; K magnitudes that grow block by
         block (the logits' running maximum moves again and again, the lazy rescale included);
      1  the same V scales with flat logits (every block carries weight);
      2  a large V scale first, small ones (1e-4 .. 1e-2) after, with growing logits: the blocks
         that dominate the softmax are the small-scale ones."""
    lens = [700, 1500, 333, 2500, 64, 1000, 17, 1234]
    w = gen.make_workload(f"p8_wide{B}", 97, 32, 8, 128, [lens[i % len(lens)] for i in range(B)])
    rng = np.random.default_rng(97)
    kf = gen.bf16_bits_to_f32(w.k_cache).copy()
    vf = gen.bf16_bits_to_f32(w.v_cache).copy()
    kn = gen.bf16_bits_to_f32(w.k_new).copy()
    vn = gen.bf16_bits_to_f32(w.v_new).copy()
    for b in range(w.B):
        nb = -(-int(w.context_lens[b]) // 16)
        kind = b % 3
        for j in range(nb):
            sk = 1.0 if kind == 1 else min(1.0 + 0.5 * j, 24.0)
            if kind == 2:
                sv = 1.0 if j == 0 else 10.0 ** rng.uniform(-4.0, -2.0)
            else:
                sv = 1e-4 if j == 0 else 10.0 ** rng.uniform(-4.0, 0.0)
            bid = int(w.block_tables[b, j])
            kf[bid] *= np.float32(sk)
            vf[bid] *= np.float32(sv)
            if j == nb - 1:
                kn[b] *= np.float32(sk)
                vn[b] *= np.float32(sv)
    return dataclasses.replace(w, k_cache=gen.f32_to_bf16_bits(kf), v_cache=gen.f32_to_bf16_bits(vf),
                               k_new=gen.f32_to_bf16_bits(kn), v_new=gen.f32_to_bf16_bits(vn))


def assert_rows_relative(got: np.ndarray, ref: np.ndarray, rel: float, what: str):
    """Each output row within rel of its own largest magnitude: the absolute tolerance says
    nothing about rows whose values are all small (the small-scale blocks dominate kind 2)."""
    scale = np.max(np.abs(ref), axis=-1)
    err = np.max(np.abs(got - ref), axis=-1)
    bad = np.argwhere(err > rel * scale)
    assert bad.size == 0, f"{what}: {len(bad)} rows beyond {rel} relative, first {bad[0].tolist()}"


@pytest.mark.parametrize("B", [6, 24], ids=["two_tiles_per_step", "one_tile_per_step"])
def test_fp8_block_scales_spanning_four_decades(pkv, oracle, B):
    """Per-(block, KV head) V scales whose ratio inside one sequence reaches 10^4 in either
    direction: every output is finite and matches the oracle, absolutely and row by row
    relative to the row's magnitude, through the single pass, fixed partitions, the fused step
    and the planner's plan (tapered partitions when the grid has a unit per SM)."""
    from paged_kv_decode_slot_gb300.step import DecodeStepFp8
    c = Fp8Case(oracle, wide_scale_workload(B), "block")
    w = c.w
    for b in range(w.B):    # the scales of one sequence's blocks span at least four decades
        vs_b = c.vs[w.block_tables[b, :-(-int(w.context_lens[b]) // 16)]]
        if vs_b.shape[0] > 40:
            assert vs_b.max() / vs_b.min() > 1e3, b
    ref, ref_lse = c.reference(oracle)
    for pb in (0, 3):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = _attn(pkv, c, c.device(appended=True), pb, err)
        assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
        got = out_f64(out)
        what = f"wide scales B={B} pb={pb}"
        assert_close(got, ref, what)
        assert_rows_relative(got, ref, 2e-2, what)
        assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, what)
        out2, lse2, _ = _step(pkv, c, c.device(appended=False), pb)
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)
    d = c.device(appended=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = DecodeStepFp8(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["k_scale"],
                         d["v_scale"], d["block_tables"], d["context_lens"], w.scale, err_flag=err)
    step.run()
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    got = out_f64(step.out)
    what = f"wide scales B={B} ({step.plan.describe()})"
    assert_close(got, ref, what)
    assert_rows_relative(got, ref, 2e-2, what)
    assert_lse_close(step.lse.cpu().numpy().astype(np.float64), ref_lse, what)
