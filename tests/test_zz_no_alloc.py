"""Split-KV attention without any allocation (GPU).

pkv_decode_attn_splitk_noalloc serves callers that cannot call cudaMalloc where they run
attention: code inside a CUDA graph capture, an allocator's own callback, or a framework
that owns the whole device heap.  It keeps its partial results in a static scratch array
built into the library instead of a caller workspace.  This test calls it through the C ABI
twice in a row, on two different batches, and checks each result against the workspace
entry point pkv_decode_attn_splitk within the attention tolerance the other tests use; it
also checks that a problem too large for the scratch is refused before anything runs.
"""
from __future__ import annotations

import pytest
import torch

from devutil import assert_close, out_f64, upload
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def _both(pkv, w, part_blocks):
    d = upload(w)
    # the decode step's append first: each sequence's newest slot holds a NaN poison until then
    slots = torch.empty(w.B, dtype=torch.int64, device="cuda")
    pkv.check(pkv.pkv_slot_mapping(d["block_tables"], d["context_lens"], w.num_blocks, slots))
    pkv.check(pkv.pkv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"]))
    P = pkv.max_partitions_for(w.max_blocks, part_blocks)
    assert pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P) <= pkv.binding.STATIC_SCRATCH_BYTES
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_na = torch.empty_like(d["q"])
    lse_na = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk_noalloc(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                                 d["context_lens"], w.scale, out_na, part_blocks, P,
                                                 lse_na, err))
    ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
    out_ws = torch.empty_like(d["q"])
    lse_ws = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, out_ws, part_blocks, P, ws,
                                         lse_ws, err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_OK, f"err_flag {flag:#x}"
    return out_na, lse_na, out_ws, lse_ws


def test_noalloc_matches_workspace_entry_point_twice(pkv):
    # two calls in a row on different batches: the second must not see the first's partials
    first = gen.make_workload("noalloc_a", 31, 32, 8, 128, gen.uniform_int(31, 9, 8, 1, 3000))
    second = gen.make_workload("noalloc_b", 32, 16, 2, 64, [1, 17, 64, 200, 513])
    for w, pb in ((first, 8), (second, 2)):
        out_na, lse_na, out_ws, lse_ws = _both(pkv, w, pb)
        assert_close(out_f64(out_na), out_f64(out_ws), f"{w.name}: no-alloc vs workspace")
        assert torch.allclose(lse_na, lse_ws, atol=2e-2, rtol=0, equal_nan=True)


def test_noalloc_refuses_problems_beyond_the_scratch(pkv):
    w = gen.make_workload("noalloc_big", 33, 32, 8, 128, [16] * 8)
    d = upload(w)
    out = torch.empty_like(d["q"])
    P = 1024           # 8 * 32 * 1024 * 128 * 4 bytes of partials: far beyond the scratch
    assert pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P) > pkv.binding.STATIC_SCRATCH_BYTES
    st = pkv.pkv_decode_attn_splitk_noalloc(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                            d["context_lens"], w.scale, out, 1, P)
    assert st == pkv.PKV_ERR_WORKSPACE
    assert "static scratch" in pkv.pkv_last_error()
