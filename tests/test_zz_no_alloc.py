"""Split-KV attention without any allocation (GPU).

pkv_decode_attn_splitk_noalloc serves callers that cannot call cudaMalloc where they run
attention: code inside a CUDA graph capture, an allocator's own callback, or a framework
that owns the whole device heap.  It keeps its partial results in a static scratch array
built into the library instead of a caller workspace.  This test calls it through the C ABI
twice in a row, on two different batches, and checks each result against the workspace
entry point pkv_decode_attn_splitk -- bit for bit, since both merge the same partials in the
same order -- and against the float64 oracle within the attention tolerance the other tests
use.  One batch has at least one (sequence, KV head) unit per SM, so its partitions taper; the
other does not.  It also checks that a problem too large for the scratch is refused before
anything runs, and that a call with no sequences (the per-device preparation) launches nothing.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from devutil import appended_host_cache, assert_close, assert_lse_close, out_f64, upload
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def _both(pkv, w, part_blocks, P):
    d = upload(w)
    # the decode step's append first: each sequence's newest slot holds a NaN poison until then
    slots = torch.empty(w.B, dtype=torch.int64, device="cuda")
    pkv.check(pkv.pkv_slot_mapping(d["block_tables"], d["context_lens"], w.num_blocks, slots))
    pkv.check(pkv.pkv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"]))
    assert pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P) <= pkv.binding.STATIC_SCRATCH_BYTES
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_na = torch.full_like(d["q"], float("nan"))
    lse_na = torch.full((w.B, w.N), float("nan"), dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk_noalloc(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                                 d["context_lens"], w.scale, out_na, part_blocks, P,
                                                 lse_na, err))
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    out_ws = torch.full_like(d["q"], float("nan"))
    lse_ws = torch.full((w.B, w.N), float("nan"), dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, out_ws, part_blocks, P, ws,
                                         lse_ws, err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_OK, f"err_flag {flag:#x}"
    return out_na, lse_na, out_ws, lse_ws


def test_noalloc_matches_workspace_entry_point_twice(pkv, oracle):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 1) at least one (sequence, KV head) unit per SM and room for the extra partition: tapered
    B = -(-sms // 8) + 8
    tapered = gen.make_workload("noalloc_a", 31, 32, 8, 128, gen.uniform_int(31, 9, B, 1, 2000))
    pb_a = 16
    P_a = pkv.tapered_partitions_for(tapered.max_blocks, pb_a)
    assert tapered.B * tapered.K >= sms and P_a > pkv.max_partitions_for(tapered.max_blocks, pb_a)
    # 2) a small batch (one wave: uniform partitions), other head shape
    small = gen.make_workload("noalloc_b", 32, 16, 2, 64, [1, 17, 64, 200, 513])
    pb_b = 2
    P_b = pkv.max_partitions_for(small.max_blocks, pb_b)
    # two calls in a row on different batches: the second must not see the first's partials
    for w, pb, P in ((tapered, pb_a, P_a), (small, pb_b, P_b)):
        out_na, lse_na, out_ws, lse_ws = _both(pkv, w, pb, P)
        assert torch.equal(out_na.view(torch.int16), out_ws.view(torch.int16)), f"{w.name}: out differs"
        assert torch.equal(lse_na, lse_ws), f"{w.name}: lse differs"
        kc, vc = appended_host_cache(oracle, w)
        ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
        assert_close(out_f64(out_na), ref, f"{w.name}: no-alloc vs oracle")
        assert_lse_close(lse_na.cpu().numpy().astype(np.float64), ref_lse, f"{w.name}: no-alloc vs oracle")


def test_noalloc_refuses_problems_beyond_the_scratch(pkv):
    w = gen.make_workload("noalloc_big", 33, 32, 8, 128, [16] * 8)
    d = upload(w)
    out = torch.full_like(d["q"], 3.0)
    P = 1024           # 8 * 32 * 1024 * 128 * 4 bytes of partials: far beyond the scratch
    assert pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P) > pkv.binding.STATIC_SCRATCH_BYTES
    st = pkv.pkv_decode_attn_splitk_noalloc(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                            d["context_lens"], w.scale, out, 1, P)
    assert st == pkv.PKV_ERR_WORKSPACE
    assert "static scratch" in pkv.pkv_last_error()
    # beyond the separate merge's partition limit, though the partials would fit: refused too
    w1 = gen.make_workload("noalloc_parts", 34, 1, 1, 64, [16])
    d1 = upload(w1)
    out1 = torch.full_like(d1["q"], 3.0)
    assert pkv.pkv_splitk_workspace_bytes(1, 1, 64, 13000) <= pkv.binding.STATIC_SCRATCH_BYTES
    st = pkv.pkv_decode_attn_splitk_noalloc(d1["q"], d1["k_cache"], d1["v_cache"], d1["block_tables"],
                                            d1["context_lens"], w1.scale, out1, 1, 13000)
    assert st == pkv.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.all(out1 == 3.0), "a refused call wrote its output"


def test_noalloc_zero_sequences_prepares_and_launches_nothing(pkv):
    """num_seqs = 0 with valid pointers: the call looks up the scratch for this device, returns
    PKV_OK and writes nothing (called through the C symbol: the binding derives num_seqs from q)."""
    import ctypes
    w = gen.make_workload("noalloc_zero", 35, 8, 2, 64, [40])
    d = upload(w)
    out = torch.full_like(d["q"], 5.0)
    lib = pkv.library()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.pkv_decode_attn_splitk_noalloc(ptr(d["q"]), ptr(d["k_cache"]), ptr(d["v_cache"]),
                                            ptr(d["block_tables"]), w.max_blocks, ptr(d["context_lens"]), 0,
                                            w.N, ctypes.c_float(w.scale), ptr(out), None,
                                            pkv.cache_desc(d["k_cache"]), 1, 4, None, None)
    assert st == pkv.PKV_OK
    torch.cuda.synchronize()
    assert torch.all(out == 5.0)
