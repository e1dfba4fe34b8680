"""Parity of the sm_103a library against the float64 oracle (GPU).

Bit-exact for slot mapping, append and gather; attention within max abs 2e-2 and mean abs
2e-3 of the oracle (bf16 inputs and output, fp32 accumulation).  Every case compares every
output element, the full-size workloads included (run in the launch configuration the
benchmark times).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from devutil import (appended_host_cache, assert_close, assert_lse_close, bf16_dev, bf16_host,
                     i32_dev, out_f64, upload)
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _no_flags(pkv, err):
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_OK and flag == 0, f"err_flag {flag:#x}"


def _post_append_device(pkv, oracle, w):
    """Upload a workload and bring its pools to the post-append state with the GPU path."""
    d = upload(w)
    slots = torch.empty(w.B, dtype=torch.int64, device="cuda")
    err = _err()
    pkv.check(pkv.pkv_slot_mapping(d["block_tables"], d["context_lens"], w.num_blocks, slots, err))
    pkv.check(pkv.pkv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"], err))
    _no_flags(pkv, err)
    d["slots"] = slots
    return d


def _single(pkv, w, d, err=None):
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                  d["context_lens"], w.scale, out, lse, err))
    return out, lse


def _splitk(pkv, w, d, part_blocks, err=None):
    P = pkv.max_partitions_for(w.max_blocks, part_blocks)
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, out, part_blocks, P, ws, lse, err))
    return out, lse


# ------------------------------------ cache operations ------------------------------------
@pytest.mark.parametrize("name", ["tiny", "l3_8b_b64", "prefix_l3_70b"])
def test_slot_mapping_and_append_bit_exact(pkv, oracle, name):
    w = gen.make_config(name)
    d = _post_append_device(pkv, oracle, w)
    assert np.array_equal(d["slots"].cpu().numpy(), oracle.slot_mapping(w.block_tables, w.context_lens))
    kc, vc = appended_host_cache(oracle, w)
    assert np.array_equal(bf16_host(d["k_cache"]), kc)
    assert np.array_equal(bf16_host(d["v_cache"]), vc)


def test_append_skips_negative_slots(pkv):
    w = gen.make_config("tiny")
    d = upload(w)
    slots = torch.tensor([-1, 5, -7, 40], dtype=torch.int64, device="cuda")
    err = _err()
    pkv.check(pkv.pkv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"], err))
    _no_flags(pkv, err)
    kc = w.k_cache.copy()
    kc[5 // 16, 5 % 16] = w.k_new[1]
    kc[40 // 16, 40 % 16] = w.k_new[3]
    assert np.array_equal(bf16_host(d["k_cache"]), kc)


@pytest.mark.parametrize("name", ["tiny", "prefix_l3_70b"])
def test_gather_bit_exact(pkv, oracle, name):
    w = gen.make_config(name)
    d = _post_append_device(pkv, oracle, w)
    kc, vc = appended_host_cache(oracle, w)
    ko, vo, cu = oracle.gather(kc, vc, w.block_tables, w.context_lens)
    rows = int(cu[-1])
    k_out = torch.empty(rows, w.K, w.H, dtype=torch.bfloat16, device="cuda")
    v_out = torch.empty_like(k_out)
    err = _err()
    pkv.check(pkv.pkv_gather(d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                             torch.from_numpy(cu[:-1].copy()).cuda(), k_out, v_out, err))
    _no_flags(pkv, err)
    assert np.array_equal(bf16_host(k_out), ko) and np.array_equal(bf16_host(v_out), vo)


# ------------------------------------ attention, small -------------------------------------
def _small_cases():
    cases = [("tiny", lambda: gen.make_config("tiny"))]
    cases.append(("ragged_gqa4_h128", lambda: gen.make_workload(
        "ragged_gqa4_h128", 7, 32, 8, 128, gen.uniform_int(7, 9, 12, 1, 2000))))
    cases.append(("mha_h128", lambda: gen.make_workload("mha_h128", 8, 8, 8, 128, [1, 15, 16, 17, 500])))
    cases.append(("gqa8_h64", lambda: gen.make_workload("gqa8_h64", 9, 16, 2, 64, [2, 31, 32, 33, 777])))
    cases.append(("gqa2_h128", lambda: gen.make_workload("gqa2_h128", 10, 8, 4, 128, [3, 48, 129, 1024])))
    cases.append(("k_scaled", lambda: gen.make_workload("k_scaled", 11, 32, 8, 128, [4096, 100], k_mult=0.5)))
    return cases


@pytest.mark.parametrize("name,make", _small_cases(), ids=[c[0] for c in _small_cases()])
def test_decode_attn_vs_oracle(pkv, oracle, name, make):
    w = make()
    d = _post_append_device(pkv, oracle, w)
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    err = _err()
    out, lse = _single(pkv, w, d, err)
    _no_flags(pkv, err)
    assert_close(out_f64(out), ref, f"{name} single-pass")
    assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name} single-pass")
    for part_blocks in (1, 2, 7):
        out_s, lse_s = _splitk(pkv, w, d, part_blocks, err)
        _no_flags(pkv, err)
        assert_close(out_f64(out_s), ref, f"{name} split-KV {part_blocks}")
        assert_lse_close(lse_s.cpu().numpy(), ref_lse, f"{name} split-KV {part_blocks}")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("H", [64, 128])
def test_decode_sweep_every_tail(pkv, oracle, G, H):
    """Context lengths 1..70: every in-block tail, one to five blocks, all group sizes."""
    K = 2
    w = gen.make_workload(f"sweep_g{G}_h{H}", 100 + G * H, G * K, K, H, list(range(1, 71)))
    d = _post_append_device(pkv, oracle, w)
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    out, lse = _single(pkv, w, d)
    assert_close(out_f64(out), ref, f"sweep G={G} H={H}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, f"sweep G={G} H={H}")
    out_s, _ = _splitk(pkv, w, d, 2)
    assert_close(out_f64(out_s), ref, f"sweep split G={G} H={H}")


def test_partitions_vs_oracle(pkv, oracle):
    w = gen.make_workload("parts", 12, 16, 4, 128, [1, 40, 200, 333])
    d = _post_append_device(pkv, oracle, w)
    kc, vc = appended_host_cache(oracle, w)
    pb = 4
    P = pkv.max_partitions_for(w.max_blocks, pb)
    po = torch.full((w.B, w.N, P, w.H), float("nan"), device="cuda")
    pl = torch.full((w.B, w.N, P), float("nan"), device="cuda")
    pkv.check(pkv.pkv_decode_attn_partitions(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                             d["context_lens"], w.scale, pb, po, pl))
    ref_po, ref_pl = oracle.decode_partitions(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                              pb * 16, P)
    po, pl = po.cpu().numpy().astype(np.float64), pl.cpu().numpy().astype(np.float64)
    for b in range(w.B):
        np_b = -(-(-(-int(w.context_lens[b]) // 16)) // pb)
        assert_close(po[b, :, :np_b], ref_po[b, :, :np_b], f"partials b={b}")
        assert_lse_close(pl[b, :, :np_b], ref_pl[b, :, :np_b], f"partial lse b={b}")
        assert np.all(np.isnan(po[b, :, np_b:])), "an empty partition was written"
    # the merge alone, fed the oracle's partials, reproduces the oracle's unsplit output
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_lse_merge(torch.from_numpy(ref_po.astype(np.float32)).cuda(),
                                torch.from_numpy(ref_pl.astype(np.float32)).cuda(),
                                d["context_lens"], pb, out, lse))
    assert_close(out_f64(out), ref, "merge of oracle partials")
    assert_lse_close(lse.cpu().numpy(), ref_lse, "merge of oracle partials")


def test_single_partition_split_is_bit_identical(pkv, oracle):
    w = gen.make_workload("p1", 13, 32, 8, 128, [1, 17, 900, 2048])
    d = _post_append_device(pkv, oracle, w)
    out, lse = _single(pkv, w, d)
    out_s, lse_s = _splitk(pkv, w, d, w.max_blocks)
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(lse, lse_s)


def test_ctx1_returns_new_v_bit_exact(pkv, oracle):
    w = gen.make_config("tiny")                 # sequence 0 has context length 1
    d = _post_append_device(pkv, oracle, w)
    out, lse = _single(pkv, w, d)
    got = bf16_host(out)[0]                     # [N, H]
    G = w.N // w.K
    for n in range(w.N):
        assert np.array_equal(got[n], w.v_new[0, n // G]), n


def test_block_permutation_bit_identical(pkv, oracle):
    w = gen.make_workload("perm", 14, 32, 8, 128, [5, 77, 300, 1500])
    d = _post_append_device(pkv, oracle, w)
    out1, lse1 = _single(pkv, w, d)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(w.num_blocks)).cuda()
    k2 = torch.empty_like(d["k_cache"])
    v2 = torch.empty_like(d["v_cache"])
    k2[perm] = d["k_cache"]
    v2[perm] = d["v_cache"]
    bt = d["block_tables"].long()
    t2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int().contiguous()
    d2 = dict(d, k_cache=k2, v_cache=v2, block_tables=t2)
    out2, lse2 = _single(pkv, w, d2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse1, lse2)


def test_ctx0_gives_zero_and_neg_inf(pkv, oracle):
    w = gen.make_workload("ctx0", 15, 8, 2, 64, [0, 20])
    d = _post_append_device(pkv, oracle, w)
    out, lse = _single(pkv, w, d)
    assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))
    out_s, lse_s = _splitk(pkv, w, d, 1)
    assert torch.all(out_s[0].float() == 0) and torch.all(torch.isneginf(lse_s[0]))
    assert float((out_s[1].float() - out[1].float()).abs().max()) <= 2e-2


# ------------------------------------ device-detected errors -------------------------------
def test_bad_block_id_sets_flag(pkv, oracle):
    w = gen.make_config("tiny")
    d = _post_append_device(pkv, oracle, w)
    for bad in (w.num_blocks, -3, 1 << 30):
        bt = d["block_tables"].clone()
        bt[3, 5] = bad
        err = _err()
        out = torch.empty_like(d["q"])
        pkv.check(pkv.pkv_decode_attn(d["q"], d["k_cache"], d["v_cache"], bt, d["context_lens"],
                                      w.scale, out, None, err))
        st, flag = pkv.pkv_read_err_flag(err)
        assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_BLOCK_RANGE
        assert torch.all(torch.isfinite(out[3].float()))   # the bad tile was skipped, not read
        slots = torch.empty(w.B, dtype=torch.int64, device="cuda")
        bt2 = d["block_tables"].clone()
        bt2[3, (int(w.context_lens[3]) - 1) // 16] = bad
        err = _err()
        pkv.check(pkv.pkv_slot_mapping(bt2, d["context_lens"], w.num_blocks, slots, err))
        st, flag = pkv.pkv_read_err_flag(err)
        assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_BLOCK_RANGE and int(slots[3]) == -1


def test_bad_slot_and_ctx_set_flags(pkv, oracle):
    w = gen.make_config("tiny")
    d = upload(w)
    before = bf16_host(d["k_cache"])
    slots = torch.tensor([w.num_blocks * 16, 1 << 40, -1, -1], dtype=torch.int64, device="cuda")
    err = _err()
    pkv.check(pkv.pkv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"], err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag == pkv.PKV_FLAG_SLOT_RANGE
    assert np.array_equal(bf16_host(d["k_cache"]), before)
    cl = d["context_lens"].clone()
    cl[2] = w.max_blocks * 16 + 1
    err = _err()
    out = torch.empty_like(d["q"])
    pkv.check(pkv.pkv_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], cl, w.scale,
                                  out, None, err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_CTX_RANGE
    assert torch.all(out[2].float() == 0)


@pytest.mark.parametrize("pb", [2, 3, 4])
def test_tapered_partitions_merge_in_kernel_and_separate(pkv, oracle, pb):
    """With at least one (sequence, KV head) unit per SM and room for one more partition, the merged
    split entry points taper their partitions (partition 0, launched last, covers half a
    partition).  Every row matches the oracle -- no block missed or counted twice for sequences
    with 0, 1, 2, 3 and many partitions, lengths on and off the half-partition edge -- and the
    in-kernel merge equals the separate merge of the same tapered partials (forced by
    max_partitions > 8192 / G) bit for bit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    K, G = 4, 4
    B = -(-sms // K) + 2
    lens = [0, 1, 16, 17, 31, 32, 33, 48, 64, 65, 80, 96, 97, 127, 128, 129, 200, 333, 700, 1000]
    w = gen.make_workload("tapered", 153, K * G, K, 128, [lens[i % len(lens)] for i in range(B)])
    assert w.B * w.K >= sms
    d = _post_append_device(pkv, oracle, w)
    # tapered partition 0 holds pb // 2 blocks (1, 1, 2), the others pb
    P = pkv.tapered_partitions_for(w.max_blocks, pb)
    assert P >= pkv.max_partitions_for(w.max_blocks, pb)
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    out_k = torch.empty_like(d["q"])
    lse_k = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, out_k, pb, P, ws, lse_k))
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out_k), ref, f"tapered split pb={pb}, in-kernel merge")
    assert_lse_close(lse_k.cpu().numpy().astype(np.float64), ref_lse, f"tapered split pb={pb}, in-kernel merge")
    P = pkv.IN_KERNEL_MERGE_WEIGHTS // G + 1
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    out_m = torch.empty_like(d["q"])
    lse_m = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, out_m, pb, P, ws, lse_m))
    torch.cuda.synchronize()
    assert torch.equal(out_k.view(torch.int16), out_m.view(torch.int16))
    assert torch.equal(lse_k, lse_m)


# ------------------------------------ full-size workloads -----------------------------------
FULL = ["l3_8b_b64", "l3_8b_b16", "l2_13b_mha_b1", "l2_13b_mha_b8", "l2_13b_mha_b64", "l2_13b_mha_b128",
        "prefix_l3_70b", "long_splitk"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(pkv, oracle, name):
    """The decode step as the benchmark times it (DecodeStep, the planner's plan, fused append) on
    every full-size workload; every sequence's output and lse against the oracle."""
    from paged_kv_decode_slot_gb300.step import DecodeStep
    w = gen.make_config(name)
    d = upload(w)
    err = _err()
    step = DecodeStep(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                      d["context_lens"], w.scale, err_flag=err)
    step.run()
    _no_flags(pkv, err)
    kc, vc = appended_host_cache(oracle, w)
    assert np.array_equal(bf16_host(d["k_cache"]), kc) and np.array_equal(bf16_host(d["v_cache"]), vc)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(step.out), ref, f"{name} ({step.plan.describe()})")
    assert_lse_close(step.lse.cpu().numpy(), ref_lse, name)


# --------------------------- partition merge paths and large shapes ---------------------------
@pytest.mark.parametrize("part_blocks", [1, 2, 7])
def test_split_merge_in_kernel_and_separate(pkv, oracle, part_blocks):
    """1-block partitions of a 20K-token sequence make 1,250 partitions: G x 1,250 weights exceed
    the attention kernel's ring, so the merge runs as a second launch; 2-block partitions (625)
    merge inside the launch.  Both, and the fused step, match the oracle; a second call on the
    same workspace (its counters back at zero) repeats the first bit for bit."""
    w = gen.make_workload("merge_paths", 151, 16, 2, 128, [20000, 3000, 1, 17])
    d = _post_append_device(pkv, oracle, w)
    out, lse = _splitk(pkv, w, d, part_blocks)
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, f"split pb={part_blocks}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"split pb={part_blocks}")
    P = pkv.max_partitions_for(w.max_blocks, part_blocks)
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        o = torch.empty_like(d["q"])
        pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                             d["context_lens"], w.scale, o, part_blocks, P, ws))
        outs.append(o)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), out.view(torch.int16))
    # the workspace counters are zero again after every call
    torch.cuda.synchronize()
    cnt_off = ws.numel() - w.B * w.N * 4
    assert int(ws[cnt_off:].view(torch.int32).abs().sum()) == 0


def test_many_short_sequences(pkv, oracle):
    """2,048 sequences of 1..64 tokens (a grid 2,048 sequences deep), every element."""
    ctx = gen.uniform_int(161, 9, 2048, 1, 64)
    w = gen.make_workload("many_short", 161, 32, 8, 128, ctx)
    d = _post_append_device(pkv, oracle, w)
    out, lse = _single(pkv, w, d)
    kc, vc = appended_host_cache(oracle, w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, "2048 short sequences")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, "2048 short sequences")


@pytest.mark.parametrize("part_blocks", [0, 4, 3])
def test_context_fills_the_table(pkv, oracle, part_blocks):
    """Every sequence as long as its table allows (ctx = max_blocks * 16): the last block is
    full and the last partition ends at the table's end (or inside it)."""
    w = gen.make_workload("full_table", 171, 16, 4, 64, [320, 320, 320], pool_factor=1.0)
    assert w.max_blocks * 16 == 320
    d = _post_append_device(pkv, oracle, w)
    out, _ = _splitk(pkv, w, d, part_blocks) if part_blocks else _single(pkv, w, d)
    kc, vc = appended_host_cache(oracle, w)
    ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, f"full tables pb={part_blocks}")


@pytest.mark.parametrize("part_blocks,H", [(3, 128), (1, 128), (2, 64), (5, 64)])
def test_in_kernel_merge_equals_separate_merge(pkv, oracle, part_blocks, H):
    """The last partition CTA's merge (inside the split launch) and lse_merge_kernel (the partials
    export followed by pkv_lse_merge) give the same bits: one merge order per row, whichever
    kernel runs it and however many rows that kernel merges at once."""
    w = gen.make_workload(f"merge_same_{H}", 152, 16, 4, H, [1, 16, 17, 300, 1000, 4000])
    d = _post_append_device(pkv, oracle, w)
    out_k, lse_k = _splitk(pkv, w, d, part_blocks)
    P = pkv.max_partitions_for(w.max_blocks, part_blocks)
    part_out = torch.empty(w.B, w.N, P, w.H, dtype=torch.float32, device="cuda")
    part_lse = torch.empty(w.B, w.N, P, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_partitions(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                             d["context_lens"], w.scale, part_blocks, part_out, part_lse))
    out_m = torch.empty_like(d["q"])
    lse_m = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_lse_merge(part_out, part_lse, d["context_lens"], part_blocks, out_m, lse_m))
    torch.cuda.synchronize()
    assert torch.equal(out_k.view(torch.int16), out_m.view(torch.int16))
    assert torch.equal(lse_k, lse_m)
