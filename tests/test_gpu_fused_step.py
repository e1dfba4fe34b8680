"""The fused decode step (pkv_decode_step) against the separate calls and the oracle (GPU).

One launch (two with partitions) must give bit for bit what slot mapping, append and attention
give as separate calls: the same output and lse, the same bytes in both pools, the same slots.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from devutil import appended_host_cache, assert_close, bf16_dev, bf16_host, i32_dev, out_f64, upload
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def _separate(pkv, w, part_blocks):
    d = upload(w)
    slots = torch.empty(w.B, dtype=torch.int64, device="cuda")
    pkv.check(pkv.pkv_slot_mapping(d["block_tables"], d["context_lens"], w.num_blocks, slots))
    pkv.check(pkv.pkv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"]))
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
        pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                             d["context_lens"], w.scale, out, part_blocks, P, ws, lse))
    else:
        pkv.check(pkv.pkv_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                      d["context_lens"], w.scale, out, lse))
    return d, out, lse, slots


def _fused(pkv, w, part_blocks, err=None):
    d = upload(w)
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
    P, ws = 0, None
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    pkv.check(pkv.pkv_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                  d["block_tables"], d["context_lens"], w.scale, out, lse, slots,
                                  part_blocks, P, ws, err))
    return d, out, lse, slots


CASES = [
    ("tiny", lambda: gen.make_config("tiny")),
    ("ragged_gqa4", lambda: gen.make_workload("f_ragged", 41, 32, 8, 128, gen.uniform_int(41, 9, 10, 1, 1500))),
    ("mha", lambda: gen.make_workload("f_mha", 42, 8, 8, 128, [1, 16, 17, 200])),
    ("gqa8_h64", lambda: gen.make_workload("f_gqa8", 43, 16, 2, 64, [31, 32, 33, 500])),
    ("prefix", lambda: gen.make_config("prefix_l3_70b")),
]


@pytest.mark.parametrize("part_blocks", [0, 2, 5])
@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_fused_step_equals_separate_calls(pkv, oracle, name, make, part_blocks):
    w = make()
    d1, out1, lse1, slots1 = _separate(pkv, w, part_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d2, out2, lse2, slots2 = _fused(pkv, w, part_blocks, err)
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_OK, f"err_flag {flag:#x}"
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    assert torch.equal(slots1, slots2)
    assert torch.equal(d1["k_cache"].view(torch.int16), d2["k_cache"].view(torch.int16))
    assert torch.equal(d1["v_cache"].view(torch.int16), d2["v_cache"].view(torch.int16))
    # and against the oracle: the pools byte for byte, the output within tolerance
    kc, vc = appended_host_cache(oracle, w)
    assert np.array_equal(bf16_host(d2["k_cache"]), kc) and np.array_equal(bf16_host(d2["v_cache"]), vc)
    assert np.array_equal(slots2.cpu().numpy(), oracle.slot_mapping(w.block_tables, w.context_lens))
    ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out2), ref, f"fused {name} pb={part_blocks}")


@pytest.mark.parametrize("G", [1, 4, 8])
def test_fused_step_every_tail(pkv, oracle, G):
    """The new token at every in-block position 0..15 and across the first blocks."""
    w = gen.make_workload(f"f_tail{G}", 50 + G, 2 * G, 2, 128, list(range(1, 50)))
    _, out1, lse1, _ = _separate(pkv, w, 0)
    _, out2, lse2, _ = _fused(pkv, w, 0)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse1, lse2)


def test_fused_step_empty_sequence_and_bad_last_block(pkv):
    w = gen.make_workload("f_edge", 60, 8, 2, 64, [0, 20, 33])
    d = upload(w)
    bt = d["block_tables"].clone()
    bt[2, 2] = w.num_blocks + 5               # sequence 2's last block (tokens 32..) is out of range
    d["block_tables"] = bt
    out = torch.empty_like(d["q"])
    slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = bf16_host(d["k_cache"])
    pkv.check(pkv.pkv_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], bt,
                                  d["context_lens"], w.scale, out, None, slots, 0, 0, None, err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_BLOCK_RANGE
    s = slots.cpu().numpy()
    assert s[0] == -1 and s[2] == -1 and s[1] == int(w.block_tables[1, 1]) * 16 + 3
    assert torch.all(out[0].float() == 0)
    after = bf16_host(d["k_cache"])
    changed = np.argwhere(np.any(after != before, axis=(2, 3)))
    assert [tuple(x) for x in changed] == [(int(w.block_tables[1, 1]), 3)]   # only sequence 1's slot


def test_packed_inputs_one_copy_per_step(pkv, oracle):
    """A step whose inputs live in one pinned staging buffer (one host->device copy per step)
    gives the same results as the step fed tensor by tensor."""
    from paged_kv_decode_slot_gb300.step import DecodeStep, PackedInputs
    w = gen.make_workload("f_packed", 77, 16, 4, 128, [30, 300, 17, 64, 900])
    d = upload(w)
    step = DecodeStep(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                      d["context_lens"], w.scale)
    packed = PackedInputs(step, step.input_names())
    assert packed.bytes_per_step() == sum(t.numel() * t.element_size() for t in step.inputs())
    q2 = gen.normal_bf16(78, 1, (w.B, w.N, w.H))
    packed.host["q"].copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16))
    packed.upload()
    step.run()
    torch.cuda.synchronize()
    ref = upload(w)
    ref_step = DecodeStep(torch.from_numpy(q2.view(np.int16)).cuda().view(torch.bfloat16), ref["k_new"],
                          ref["v_new"], ref["k_cache"], ref["v_cache"], ref["block_tables"],
                          ref["context_lens"], w.scale)
    ref_step.run()
    torch.cuda.synchronize()
    assert torch.equal(step.out.view(torch.int16), ref_step.out.view(torch.int16))
    assert torch.equal(step.k_cache.view(torch.int16), ref_step.k_cache.view(torch.int16))


def test_layer_stack_graph_replay_equals_eager(pkv, oracle):
    """A three-layer decode step (each layer its own pools and q / k_new / v_new, the same block
    tables and context lengths): one CUDA-graph replay equals the eager layer-by-layer launches
    bit for bit, and every layer matches the oracle on its own pools."""
    from paged_kv_decode_slot_gb300.step import DecodeStep, LayerStack, StepGraph, plan_attention
    L = 3
    base = gen.make_workload("layers", 171, 16, 4, 128, [1, 17, 300, 1500, 64])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = plan_attention(base.B, base.K, base.max_blocks, sms, partition_blocks=32)

    def layer_inputs(l):
        # layer l: its own K/V history and new rows (distinct draws), the same sequences
        kc = gen.normal_bf16(171, 10 + l, base.k_cache.shape)
        vc = gen.normal_bf16(171, 20 + l, base.v_cache.shape)
        q = gen.normal_bf16(171, 30 + l, base.q.shape)
        kn = gen.normal_bf16(171, 40 + l, base.k_new.shape)
        vn = gen.normal_bf16(171, 50 + l, base.v_new.shape)
        return q, kn, vn, kc, vc

    host = [layer_inputs(l) for l in range(L)]
    bt, cl = i32_dev(base.block_tables), i32_dev(base.context_lens)

    def make_stack():
        return LayerStack([DecodeStep(bf16_dev(q), bf16_dev(kn), bf16_dev(vn), bf16_dev(kc), bf16_dev(vc), bt, cl,
                                      base.scale, plan=plan) for q, kn, vn, kc, vc in host])

    eager = make_stack()
    eager.run()
    graphed = make_stack()
    g = StepGraph(graphed)
    g.replay()
    torch.cuda.synchronize()
    slots = oracle.slot_mapping(base.block_tables, base.context_lens)
    for l, (q, kn, vn, kc, vc) in enumerate(host):
        a, b = eager.layers[l], graphed.layers[l]
        assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16)), l
        assert torch.equal(a.lse, b.lse) and torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
        kc2, vc2 = kc.copy(), vc.copy()
        oracle.append(kn, vn, slots, kc2, vc2)
        ref, _ = oracle.decode(q, kc2, vc2, base.block_tables, base.context_lens, base.scale)
        assert_close(out_f64(b.out), ref, f"layer {l}")


@pytest.mark.parametrize("part_blocks", [0, 32])
def test_step_with_host_resident_inputs_and_outputs(pkv, oracle, part_blocks):
    """q, k_new, v_new, block tables, context lengths, out, lse and the slot mapping in pinned host
    memory (read and written by the kernel in place), the pools in HBM: the same bits as with
    every buffer on the device."""
    from paged_kv_decode_slot_gb300.step import AttentionPlan, DecodeStep
    w = gen.make_workload("hostio", 181, 32, 8, 128, [1, 17, 300, 2000, 64, 900])
    P = pkv.max_partitions_for(w.max_blocks, part_blocks) if part_blocks else 1
    plan = AttentionPlan("split", part_blocks, P) if part_blocks else AttentionPlan("single")

    def pinned(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(dt)).pin_memory()

    d = upload(w)
    dev_step = DecodeStep(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], w.scale, plan=plan)
    dev_step.run()
    h = upload(w)
    host_step = DecodeStep(pinned(w.q, np.int16).view(torch.bfloat16), pinned(w.k_new, np.int16).view(torch.bfloat16),
                           pinned(w.v_new, np.int16).view(torch.bfloat16), h["k_cache"], h["v_cache"],
                           pinned(w.block_tables, np.int32), pinned(w.context_lens, np.int32), w.scale, plan=plan)
    host_step.out = torch.empty(tuple(dev_step.out.shape), dtype=torch.bfloat16).pin_memory()
    host_step.lse = torch.empty(tuple(dev_step.lse.shape), dtype=torch.float32).pin_memory()
    host_step.slot_mapping = torch.empty(tuple(dev_step.slot_mapping.shape), dtype=torch.int64).pin_memory()
    host_step.run()
    torch.cuda.synchronize()
    assert torch.equal(dev_step.out.cpu().view(torch.int16), host_step.out.view(torch.int16))
    assert torch.equal(dev_step.lse.cpu(), host_step.lse)
    assert torch.equal(dev_step.slot_mapping.cpu(), host_step.slot_mapping)
    assert torch.equal(d["k_cache"].view(torch.int16), h["k_cache"].view(torch.int16))  # NaN-poisoned pools:
    assert torch.equal(d["v_cache"].view(torch.int16), h["v_cache"].view(torch.int16))  # compare the bits
