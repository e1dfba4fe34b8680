"""Several new tokens per sequence, shared-prefix decode and copy-on-write, on the GPU.

Multi-token decode (speculative verification): slots bit-exact, attention within the bf16
tolerance of the oracle's masked attention, T = 1 bit-identical to the one-token kernel.  With
more than 16 query rows per CTA (T * G, in chunks of 32) at H = 128 the tcgen05 column kernel runs:
T = 8, 9 at G = 4 and T = 3 and up at G = 8 (rows 24 .. 72, partial chunks); fewer rows and H = 64
run the mma.sync column kernel.
Shared-prefix decode: within tolerance of the oracle's plain decode (the prefix pass plus suffix
pass plus merge reach the same definition).  Block copies: bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from devutil import (appended_host_cache, assert_close, assert_lse_close, bf16_dev, bf16_host, i32_dev,
                     out_f64, upload)
from paged_kv_decode_slot_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


class MultiCase:
    """A workload whose sequences each end with T new tokens, appended by the oracle."""

    def __init__(self, oracle, w: gen.Workload, T: int, seed: int):
        self.w, self.T = w, T
        self.k_new = gen.normal_bf16(seed, 700, (w.B, T, w.K, w.H))
        self.v_new = gen.normal_bf16(seed, 701, (w.B, T, w.K, w.H))
        self.q = gen.normal_bf16(seed, 702, (w.B, T, w.N, w.H))
        self.slots = oracle.slot_mapping_multi(w.block_tables, w.context_lens, T)
        self.kc, self.vc = w.k_cache.copy(), w.v_cache.copy()
        oracle.append(self.k_new.reshape(-1, w.K, w.H), self.v_new.reshape(-1, w.K, w.H),
                      self.slots.reshape(-1), self.kc, self.vc)

    def reference(self, oracle):
        w = self.w
        return oracle.decode_multi(self.q, self.kc, self.vc, w.block_tables, w.context_lens, w.scale)


def run_multi(pkv, c: MultiCase, kc, vc, part_blocks, err=None):
    w = c.w
    q = bf16_dev(c.q)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, c.T, w.N, dtype=torch.float32, device="cuda")
    P, ws = 0, None
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B * c.T, w.N, w.H, P), dtype=torch.uint8,
                         device="cuda")
    pkv.check(pkv.pkv_decode_attn_multi(q, kc, vc, i32_dev(w.block_tables), i32_dev(w.context_lens),
                                        w.scale, out, lse, part_blocks, P, ws, err))
    return out, lse


MULTI_CASES = [
    # (name, N, K, H, context lengths) -- lengths below T, at block edges and long ones
    ("gqa4_h128", 16, 4, 128, [1, 2, 3, 4, 5, 15, 16, 17, 33, 250, 700]),
    ("gqa8_h128", 16, 2, 128, [3, 8, 16, 31, 64, 300]),
    ("mha_h64", 4, 4, 64, [2, 9, 16, 17, 129]),
    ("gqa2_h64", 8, 4, 64, [4, 20, 47]),
]


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_slot_mapping_multi_matches_oracle(pkv, oracle, T):
    w = gen.make_workload("m_slots", 70 + T, 8, 2, 64, [1, 2, 15, 16, 17, 40, 100])
    slots = torch.full((w.B, T), -7, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_slot_mapping_multi(i32_dev(w.block_tables), i32_dev(w.context_lens), w.num_blocks,
                                         slots, err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert np.array_equal(slots.cpu().numpy(), oracle.slot_mapping_multi(w.block_tables, w.context_lens, T))


@pytest.mark.parametrize("part_blocks", [0, 2, 5])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 8, 9])
@pytest.mark.parametrize("name,N,K,H,ctx", MULTI_CASES, ids=[c[0] for c in MULTI_CASES])
def test_decode_attn_multi_matches_oracle(pkv, oracle, name, N, K, H, ctx, T, part_blocks):
    w = gen.make_workload(f"m_{name}", 80 + T, N, K, H, ctx)
    c = MultiCase(oracle, w, T, 90 + T)
    # the device append path: multi-token slot mapping, then the ordinary append
    d = upload(w)
    slots = torch.empty(w.B, T, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_slot_mapping_multi(d["block_tables"], d["context_lens"], w.num_blocks, slots, err))
    pkv.check(pkv.pkv_append(bf16_dev(c.k_new.reshape(-1, K, H)), bf16_dev(c.v_new.reshape(-1, K, H)),
                             slots.reshape(-1), d["k_cache"], d["v_cache"], err))
    assert np.array_equal(bf16_host(d["k_cache"]), c.kc) and np.array_equal(bf16_host(d["v_cache"]), c.vc)
    out, lse = run_multi(pkv, c, d["k_cache"], d["v_cache"], part_blocks, err)
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(out), ref, f"multi {name} T={T} pb={part_blocks}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"multi {name} T={T} pb={part_blocks}")


@pytest.mark.parametrize("T,N,K,H", [(8, 16, 4, 128), (9, 16, 4, 128), (2, 16, 4, 128), (4, 4, 4, 64)],
                         ids=["tcgen05_T8", "tcgen05_T9_two_chunks", "mma_T2", "mma_mha_h64_T4"])
def test_multi_in_kernel_merge_equals_separate_merge(pkv, oracle, T, N, K, H):
    """Partitioned multi-token attention with the merge its kernel picks (mma.sync: by the last CTA
    of each (sequence, KV head, chunk) in the same launch; tcgen05: pkv_lse_merge) equals the same
    partials merged by pkv_lse_merge (forced by a max_partitions whose 32 x max_partitions weights
    exceed the in-kernel budget), bit for bit -- with an empty sequence, sequences shorter than T,
    single-partition sequences written out directly, and a second call on the same workspace (the
    counters were left at zero)."""
    w = gen.make_workload(f"m_merge_{T}", 300 + T, N, K, H, [0, 1, T - 1, 16, 17, 40, 333, 700, 1000])
    c = MultiCase(oracle, w, T, 310 + T)
    kc, vc = bf16_dev(c.kc), bf16_dev(c.vc)
    pb = 8
    P = pkv.max_partitions_for(w.max_blocks, pb)
    assert 32 * P <= pkv.IN_KERNEL_MERGE_WEIGHTS < 32 * 300
    q = bf16_dev(c.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for parts, calls in ((P, 2), (300, 1)):
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B * T, N, H, parts), dtype=torch.uint8, device="cuda")
        for _ in range(calls):
            out = torch.full_like(q, float("nan"))
            lse = torch.full((w.B, T, N), float("nan"), dtype=torch.float32, device="cuda")
            pkv.check(pkv.pkv_decode_attn_multi(q, kc, vc, i32_dev(w.block_tables), i32_dev(w.context_lens),
                                                w.scale, out, lse, pb, parts, ws, err))
            outs.append((out, lse))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    (o1, l1), (o2, l2), (o3, l3) = outs
    assert torch.equal(o1, o3) and torch.equal(l1, l3), "in-kernel merge differs from pkv_lse_merge"
    assert torch.equal(o1, o2) and torch.equal(l1, l2), "second call on the same workspace differs"
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(o1), ref, f"multi in-kernel merge T={T}")
    assert_lse_close(l1.cpu().numpy().astype(np.float64), ref_lse, f"multi in-kernel merge T={T}")


@pytest.mark.parametrize("T,pb", [(2, 4), (4, 4), (4, 3)])
def test_multi_tapered_partitions(pkv, oracle, T, pb):
    """With at least one (sequence, chunk, KV head) unit per SM and room for one more partition the
    mma.sync column kernel tapers its partitions (partition 0, launched last, covers half a
    partition).  Every row matches the oracle -- 0, 1, 2, 3 and many partitions, lengths on and
    off the half-partition edge, lengths below T -- and the in-kernel merge equals pkv_lse_merge of
    the same tapered partials (forced by 32 x max_partitions > 8192) bit for bit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    K, G = 4, 4
    B = -(-sms // K) + 2
    lens = [0, 1, T - 1, 16, 17, 31, 32, 33, 48, 64, 65, 96, 97, 127, 128, 129, 200, 333, 700, 1000]
    w = gen.make_workload(f"m_taper_{T}", 320 + T, K * G, K, 128, [lens[i % len(lens)] for i in range(B)])
    assert w.B * w.K >= sms and not pkv.pkv_multi_uses_tcgen05(T, w.N, w.K, w.H)
    c = MultiCase(oracle, w, T, 330 + T)
    kc, vc = bf16_dev(c.kc), bf16_dev(c.vc)
    q = bf16_dev(c.q)
    P = pkv.tapered_partitions_for(w.max_blocks, pb)
    assert P >= pkv.max_partitions_for(w.max_blocks, pb)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for parts in (P, 300):
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B * T, w.N, w.H, parts), dtype=torch.uint8, device="cuda")
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, T, w.N), float("nan"), dtype=torch.float32, device="cuda")
        pkv.check(pkv.pkv_decode_attn_multi(q, kc, vc, i32_dev(w.block_tables), i32_dev(w.context_lens),
                                            w.scale, out, lse, pb, parts, ws, err))
        outs.append((out, lse))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    (o1, l1), (o2, l2) = outs
    assert torch.equal(o1, o2) and torch.equal(l1, l2), "in-kernel merge differs from pkv_lse_merge"
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(o1), ref, f"multi tapered T={T}")
    assert_lse_close(l1.cpu().numpy().astype(np.float64), ref_lse, f"multi tapered T={T}")


@pytest.mark.parametrize("part_blocks", [0, 3])
def test_multi_with_one_token_is_the_decode_kernel(pkv, oracle, part_blocks):
    """T = 1 through the column-parallel kernel equals pkv_decode_attn / _splitk bit for bit."""
    w = gen.make_workload("m_t1", 99, 32, 8, 128, gen.uniform_int(99, 9, 10, 1, 900))
    kc, vc = appended_host_cache(oracle, w)
    dk, dv = bf16_dev(kc), bf16_dev(vc)
    q = bf16_dev(w.q)
    bt, cl = i32_dev(w.block_tables), i32_dev(w.context_lens)
    out1 = torch.empty_like(q)
    lse1 = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    out2 = torch.empty(w.B, 1, w.N, w.H, dtype=torch.bfloat16, device="cuda")
    lse2 = torch.empty(w.B, 1, w.N, dtype=torch.float32, device="cuda")
    if part_blocks:
        P = pkv.max_partitions_for(w.max_blocks, part_blocks)
        ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B, w.N, w.H, P), dtype=torch.uint8, device="cuda")
        pkv.check(pkv.pkv_decode_attn_splitk(q, dk, dv, bt, cl, w.scale, out1, part_blocks, P, ws, lse1))
        ws2 = torch.zeros_like(ws)  # zeroed before its first use, like every split workspace
        pkv.check(pkv.pkv_decode_attn_multi(q.view(w.B, 1, w.N, w.H), dk, dv, bt, cl, w.scale, out2, lse2,
                                            part_blocks, P, ws2))
    else:
        pkv.check(pkv.pkv_decode_attn(q, dk, dv, bt, cl, w.scale, out1, lse1))
        pkv.check(pkv.pkv_decode_attn_multi(q.view(w.B, 1, w.N, w.H), dk, dv, bt, cl, w.scale, out2, lse2))
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(w.B, w.N, w.H).view(torch.int16))
    assert torch.equal(lse1, lse2.view(w.B, w.N))


def test_multi_full_size_every_row(pkv, oracle):
    """Llama-3-8B-shaped batch of 64 verifying 4 tokens each (gamma = 3), one pass and partitions."""
    w = gen.make_config("l3_8b_b64")
    T = 4
    c = MultiCase(oracle, w, T, 123)
    kc, vc = bf16_dev(c.kc), bf16_dev(c.vc)
    out, _ = run_multi(pkv, c, kc, vc, 0)
    out_s, _ = run_multi(pkv, c, kc, vc, 64)
    # the multi-token step's own plan: 128-block partitions, tapered (512 units cover the SMs)
    from paged_kv_decode_slot_gb300.step import MultiTokenStep
    step = MultiTokenStep(bf16_dev(c.q), bf16_dev(c.k_new), bf16_dev(c.v_new), kc, vc, i32_dev(w.block_tables),
                          i32_dev(w.context_lens), w.scale)
    assert step.plan.mode == "split"
    assert step.plan.max_partitions == pkv.tapered_partitions_for(w.max_blocks, step.plan.partition_blocks)
    step.attention()
    ref, _ = c.reference(oracle)
    assert_close(out_f64(out), ref, "multi l3_8b_b64 one pass")
    assert_close(out_f64(out_s), ref, "multi l3_8b_b64 partitions")
    assert_close(out_f64(step.out), ref, "multi l3_8b_b64 step plan (tapered)")


# ------------------------------------ copy-on-write ----------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_copy_blocks_matches_oracle(pkv, oracle, dtype):
    w = gen.make_workload("cow", 111, 8, 2, 128, [20, 40, 9, 70], pool_blocks=40)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    if dtype == "e4m3":
        kc = (kc & 0xFF).astype(np.uint8)
        vc = (vc >> 8).astype(np.uint8)
    rng = np.random.default_rng(3)
    perm = rng.permutation(w.num_blocks)
    pairs = np.stack([perm[:10], perm[10:20]], axis=1).astype(np.int32)  # sources and distinct targets
    ref_k, ref_v = kc.copy(), vc.copy()
    oracle.copy_blocks(ref_k, ref_v, pairs)
    if dtype == "bf16":
        dk, dv = bf16_dev(kc), bf16_dev(vc)
    else:
        dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_copy_blocks(dk, dv, i32_dev(pairs), err))
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    got_k = bf16_host(dk) if dtype == "bf16" else dk.cpu().numpy()
    got_v = bf16_host(dv) if dtype == "bf16" else dv.cpu().numpy()
    assert np.array_equal(got_k, ref_k) and np.array_equal(got_v, ref_v)
    # an id outside the pool is flagged and skipped
    bad = i32_dev(np.array([[0, w.num_blocks]], dtype=np.int32))
    pkv.check(pkv.pkv_copy_blocks(dk, dv, bad, err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_BLOCK_RANGE


def test_copy_on_write_split_keeps_attention(pkv, oracle):
    """Give every sequence of the shared-prefix batch a private copy of one shared block and point
    its table there: attention is bit-identical."""
    w = gen.make_config("prefix_l3_70b")
    kc, vc = appended_host_cache(oracle, w)
    dk, dv = bf16_dev(kc), bf16_dev(vc)
    q = bf16_dev(w.q)
    bt, cl = i32_dev(w.block_tables), i32_dev(w.context_lens)
    out1 = torch.empty_like(q)
    pkv.check(pkv.pkv_decode_attn(q, dk, dv, bt, cl, w.scale, out1))
    used = set(w.block_tables[w.block_tables >= 0].tolist()) | {w.notes["orig_partial_block"]}
    free = [x for x in range(w.num_blocks) if x not in used][:w.B]
    assert len(free) == w.B
    src = int(w.block_tables[0, 5])
    pairs = np.array([[src, f] for f in free], dtype=np.int32)
    pkv.check(pkv.pkv_copy_blocks(dk, dv, i32_dev(pairs)))
    tables = w.block_tables.copy()
    tables[:, 5] = free
    out2 = torch.empty_like(q)
    pkv.check(pkv.pkv_decode_attn(q, dk, dv, i32_dev(tables), cl, w.scale, out2))
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


# ------------------------------------ shared prefixes --------------------------------------
def share_prefixes(w: gen.Workload, groups):
    """Rewrite the tables so that each group's members use the first member's leading blocks.
    groups: (start, end, prefix_blocks); every member keeps prefix_blocks * 16 < ctx."""
    tables = w.block_tables.copy()
    starts, pblocks = [0], []
    for s, e, p in groups:
        assert starts[-1] <= s
        if starts[-1] < s:                 # sequences between groups form a group without prefix
            pblocks.append(0)
            starts.append(s)
        for b in range(s, e):
            assert p * 16 < int(w.context_lens[b])
            tables[b, :p] = tables[s, :p]
        pblocks.append(p)
        starts.append(e)
    if starts[-1] < w.B:
        pblocks.append(0)
        starts.append(w.B)
    return tables, np.array(starts, dtype=np.int32), np.array(pblocks, dtype=np.int32)


def run_prefix(pkv, w, kc, vc, tables, starts, pblocks, part_blocks, max_group=None, max_prefix=None,
               err=None, prefix_part_blocks=0):
    q = bf16_dev(w.q)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    max_group = max_group or int(np.max(np.diff(starts)))
    max_prefix = int(pblocks.max()) if max_prefix is None else max_prefix
    ws = torch.empty(pkv.pkv_prefix_workspace_bytes(w.B, w.N, w.H, tables.shape[1], max_prefix, part_blocks,
                                                    prefix_part_blocks),
                     dtype=torch.uint8, device="cuda")
    pkv.check(pkv.pkv_decode_attn_prefix(q, kc, vc, i32_dev(tables), i32_dev(w.context_lens), w.scale,
                                         i32_dev(starts), i32_dev(pblocks), max_group, max_prefix, out, lse,
                                         part_blocks, ws, err, prefix_partition_blocks=prefix_part_blocks))
    return out, lse


@pytest.mark.parametrize("part_blocks,prefix_part_blocks", [(4, 0), (8, 0), (16, 0), (64, 0), (16, 4), (8, 2),
                                                           (16, 7)])
def test_prefix_workload_matches_oracle(pkv, oracle, part_blocks, prefix_part_blocks):
    w = gen.make_config("prefix_l3_70b")
    starts, pblocks = w.prefix_groups()
    kc, vc = appended_host_cache(oracle, w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefix(pkv, w, bf16_dev(kc), bf16_dev(vc), w.block_tables, starts, pblocks, part_blocks,
                          err=err, prefix_part_blocks=prefix_part_blocks)
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, f"prefix pb={part_blocks}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"prefix pb={part_blocks}")


PREFIX_CASES = [
    # name, N, K, H, context lengths, groups (start, end, shared blocks)
    ("two_groups_gqa4", 32, 8, 128, [200, 300, 180, 500, 90, 64, 700, 40],
     [(0, 3, 11), (3, 7, 3)]),
    ("singles_between", 16, 2, 128, [100, 120, 17, 300, 260, 33, 35], [(0, 2, 6), (3, 5, 16)]),
    ("mha_h64", 8, 8, 64, [70, 90, 110, 130, 150], [(0, 5, 4)]),
    ("big_group_g8", 64, 8, 128, [130 + 7 * i for i in range(12)], [(0, 12, 8)]),  # 96 rows: 3 chunks
]


@pytest.mark.parametrize("part_blocks,prefix_part_blocks", [(2, 0), (5, 0), (16, 0), (16, 3)])
@pytest.mark.parametrize("name,N,K,H,ctx,groups", PREFIX_CASES, ids=[c[0] for c in PREFIX_CASES])
def test_prefix_groups_match_oracle(pkv, oracle, name, N, K, H, ctx, groups, part_blocks, prefix_part_blocks):
    w = gen.make_workload(f"p_{name}", 131, N, K, H, ctx)
    tables, starts, pblocks = share_prefixes(w, groups)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    slots = oracle.slot_mapping(tables, w.context_lens)
    oracle.append(w.k_new, w.v_new, slots, kc, vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefix(pkv, w, bf16_dev(kc), bf16_dev(vc), tables, starts, pblocks, part_blocks, err=err,
                          prefix_part_blocks=prefix_part_blocks)
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref, ref_lse = oracle.decode(w.q, kc, vc, tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, f"prefix {name} pb={part_blocks}")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"prefix {name} pb={part_blocks}")


def test_prefix_bounds_are_flagged(pkv, oracle):
    w = gen.make_workload("p_bounds", 141, 16, 4, 128, [100, 120, 140, 160])
    tables, starts, pblocks = share_prefixes(w, [(0, 4, 5)])
    kc, vc = appended_host_cache(oracle, w)
    dk, dv = bf16_dev(kc), bf16_dev(vc)
    # a group larger than the declared bound
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_prefix(pkv, w, dk, dv, tables, starts, pblocks, 4, max_group=1, err=err)
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_GROUP_RANGE
    # a member shorter than its group's prefix
    err.zero_()
    bad = pblocks.copy()
    bad[0] = 7                         # 112 tokens > ctx of sequence 0 (100)
    out, _ = run_prefix(pkv, w, dk, dv, tables, starts, bad, 4, err=err)
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag & pkv.PKV_FLAG_GROUP_RANGE
    assert torch.all(out[0].float() == 0)


@pytest.mark.parametrize("T", [8, 4])
def test_multi_step_full_size_in_bench_plan(pkv, oracle, T):
    """The multi-token step as the benchmark times it (MultiTokenStep with its default plan) on the
    Llama-3-8B-shaped batch of 64: T = 8 and T = 4 new tokens (32 query rows per CTA: the tcgen05
    column kernel; 16: the mma.sync one), every sequence against the oracle."""
    from paged_kv_decode_slot_gb300.step import MultiTokenStep
    w = gen.make_config("l3_8b_b64")
    c = MultiCase(oracle, w, T, 200 + T)
    kc, vc = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = MultiTokenStep(bf16_dev(c.q), bf16_dev(c.k_new), bf16_dev(c.v_new), kc, vc, i32_dev(w.block_tables),
                          i32_dev(w.context_lens), w.scale, err_flag=err)
    step.run()
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(step.out), ref, f"multi step T={T} ({step.plan.describe()})")
    assert_lse_close(step.lse.cpu().numpy().astype(np.float64), ref_lse, f"multi step T={T}")


def test_multi_skipped_block_is_flagged_and_masked(pkv, oracle):
    """An out-of-range block id in one sequence's table (tcgen05 path, T = 8, G = 4): the range
    flag is raised, the tile is skipped, and every other sequence still matches the oracle."""
    w = gen.make_workload("m_badblk", 131, 16, 4, 128, [40, 90, 300, 17])
    T = 8
    c = MultiCase(oracle, w, T, 132)
    bt = w.block_tables.copy()
    bt[2, 3] = w.num_blocks + 5
    out, lse = None, None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = bf16_dev(c.q)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, T, w.N, dtype=torch.float32, device="cuda")
    pkv.check(pkv.pkv_decode_attn_multi(q, bf16_dev(c.kc), bf16_dev(c.vc), i32_dev(bt), i32_dev(w.context_lens),
                                        w.scale, out, lse, 0, 0, None, err))
    code, flags = pkv.pkv_read_err_flag(err)
    assert flags & pkv.PKV_FLAG_BLOCK_RANGE
    ref, _ = c.reference(oracle)
    keep = [0, 1, 3]
    assert_close(out_f64(out)[keep], ref[keep], "multi with a skipped block, other sequences")


# ------------------------------- fused multi-token step -------------------------------------
FUSED_CASES = [
    # (T, N, K, H, plan): plan "one_pass", "split" (uniform partitions) or "tapered"
    (2, 16, 4, 128, "one_pass"), (4, 16, 4, 128, "split"), (4, 16, 4, 128, "tapered"),
    (8, 16, 4, 128, "one_pass"), (8, 16, 4, 128, "split"), (9, 16, 4, 128, "split"),
    (3, 8, 4, 64, "split"), (20, 4, 4, 64, "one_pass"),
]


@pytest.mark.parametrize("T,N,K,H,plan", FUSED_CASES,
                         ids=[f"T{c[0]}_G{c[1] // c[2]}_H{c[3]}_{c[4]}" for c in FUSED_CASES])
def test_fused_multi_step_equals_separate_calls(pkv, oracle, T, N, K, H, plan):
    """pkv_decode_step_multi (the producers write the new rows into the pools before loading their
    blocks) equals pkv_slot_mapping_multi + pkv_append + pkv_decode_attn_multi bit for bit: out,
    lse, slots, both pools and the error flags -- with an empty sequence, contexts shorter than T,
    new tokens that straddle a block edge, and (in the tapered case) enough units to taper -- and
    matches the oracle.  T = 8, 9 at G = 4 run the tcgen05 column kernel, the rest mma.sync."""
    lens = [0, 1, T - 1, T, T + 1, 15, 16, 17, 33, 300, 700, 1000]
    B = len(lens)
    if plan == "tapered":
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        B = -(-sms // K) + 2
    w = gen.make_workload(f"fused_m_{T}_{plan}", 500 + T, N, K, H, [lens[i % len(lens)] for i in range(B)])
    c = MultiCase(oracle, w, T, 510 + T)
    pb = 0 if plan == "one_pass" else 4
    P = 0
    if plan == "split":
        P = pkv.max_partitions_for(w.max_blocks, pb)
    elif plan == "tapered":
        P = pkv.tapered_partitions_for(w.max_blocks, pb)
        assert w.B * w.K >= torch.cuda.get_device_properties(0).multi_processor_count
    q, kn, vn = bf16_dev(c.q), bf16_dev(c.k_new), bf16_dev(c.v_new)
    bt, cl = i32_dev(w.block_tables), i32_dev(w.context_lens)
    res = []
    for fused in (False, True):
        kc, vc = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, T, N), float("nan"), dtype=torch.float32, device="cuda")
        slots = torch.full((w.B, T), -7, dtype=torch.int64, device="cuda")
        ws = None
        if P:
            ws = torch.zeros(pkv.pkv_splitk_workspace_bytes(w.B * T, N, H, P), dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            pkv.check(pkv.pkv_decode_step_multi(q, kn, vn, kc, vc, bt, cl, w.scale, out, lse, slots, pb, P, ws, err))
        else:
            pkv.check(pkv.pkv_slot_mapping_multi(bt, cl, w.num_blocks, slots, err))
            pkv.check(pkv.pkv_append(kn.view(-1, K, H), vn.view(-1, K, H), slots.view(-1), kc, vc, err))
            pkv.check(pkv.pkv_decode_attn_multi(q, kc, vc, bt, cl, w.scale, out, lse, pb, P, ws, err))
        res.append((out, lse, slots, kc, vc, pkv.pkv_read_err_flag(err)))
    (o1, l1, s1, k1, v1, f1), (o2, l2, s2, k2, v2, f2) = res
    assert f1 == f2 == (pkv.PKV_OK, 0)
    assert torch.equal(s1, s2) and np.array_equal(s2.cpu().numpy(), c.slots)
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16)) and torch.equal(v1.view(torch.int16),
                                                                                   v2.view(torch.int16))
    assert np.array_equal(bf16_host(k2), c.kc) and np.array_equal(bf16_host(v2), c.vc)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    ref, ref_lse = c.reference(oracle)
    assert_close(out_f64(o2), ref, f"fused multi T={T} {plan}")
    assert_lse_close(l2.cpu().numpy().astype(np.float64), ref_lse, f"fused multi T={T} {plan}")


@pytest.mark.parametrize("T", [4, 8])
def test_fused_multi_step_bad_block_is_flagged_and_skipped(pkv, oracle, T):
    """A table entry outside the pool in the block that holds the new tokens: flagged, slots -1,
    nothing written there, the tile skipped -- as the separate calls do -- and every other
    sequence matches the oracle."""
    w = gen.make_workload(f"fused_bad_{T}", 520 + T, 16, 4, 128, [40, 90, 300, 17])
    c = MultiCase(oracle, w, T, 530 + T)
    bt_np = w.block_tables.copy()
    bt_np[2, (int(w.context_lens[2]) - 1) // 16] = w.num_blocks + 5
    q, kn, vn = bf16_dev(c.q), bf16_dev(c.k_new), bf16_dev(c.v_new)
    bt, cl = i32_dev(bt_np), i32_dev(w.context_lens)
    res = []
    for fused in (False, True):
        kc, vc = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
        out = torch.empty_like(q)
        slots = torch.full((w.B, T), -7, dtype=torch.int64, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            pkv.check(pkv.pkv_decode_step_multi(q, kn, vn, kc, vc, bt, cl, w.scale, out, None, slots, 0, 0, None,
                                                err))
        else:
            pkv.check(pkv.pkv_slot_mapping_multi(bt, cl, w.num_blocks, slots, err))
            pkv.check(pkv.pkv_append(kn.view(-1, 4, 128), vn.view(-1, 4, 128), slots.view(-1), kc, vc, err))
            pkv.check(pkv.pkv_decode_attn_multi(q, kc, vc, bt, cl, w.scale, out, None, 0, 0, None, err))
        res.append((out, slots, kc, vc, pkv.pkv_read_err_flag(err)))
    (o1, s1, k1, v1, f1), (o2, s2, k2, v2, f2) = res
    assert f1 == f2 and f2[1] & pkv.PKV_FLAG_BLOCK_RANGE
    assert torch.equal(s1, s2) and torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    ref, _ = c.reference(oracle)
    keep = [0, 1, 3]
    assert_close(out_f64(o2)[keep], ref[keep], "fused multi with a bad block, other sequences")


@pytest.mark.parametrize("prefix_part_blocks", [64, 128])
def test_prefix_long_cascade_matches_oracle(pkv, oracle, prefix_part_blocks):
    """20 sequences sharing a 32,008-token prompt (2,000 full shared blocks, about the L2's size in
    K/V): the cascade (the prefix pass on the tcgen05 column kernel, 160 query rows per KV head in
    chunks of 32) matches the oracle's plain decode on every row."""
    w = gen.make_config("prefix_long_l3_70b")
    starts, pblocks = w.prefix_groups()
    assert int(pblocks[0]) == 2000
    kc, vc = appended_host_cache(oracle, w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_prefix(pkv, w, bf16_dev(kc), bf16_dev(vc), w.block_tables, starts, pblocks, 16, err=err,
                          prefix_part_blocks=prefix_part_blocks)
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, f"long prefix, {prefix_part_blocks}-block prefix partitions")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse, "long prefix")


# ------------------------------- fused shared-prefix step -------------------------------------
FUSED_PREFIX_CASES = [
    # name, N, K, H, context lengths, groups (start, end, shared blocks).  Rows of a group = members
    # x G: up to 16 on mma.sync (both passes in one launch), 17..32 on the 32-row tcgen05 prefix pass,
    # more on the 128-row one (the suffix pass then a second launch, overlapping the first)
    ("mma_two_groups_empty_single", 16, 2, 128, [100, 120, 0, 300, 260, 33, 35], [(0, 2, 6), (3, 5, 16)]),
    ("tc32_g8", 64, 8, 128, [150, 170, 190, 210, 77], [(0, 4, 9)]),
    ("tc128_g8_edges", 64, 8, 128, [130 + 7 * i for i in range(11)] + [129], [(0, 12, 8)]),
    ("tc128_long_suffix", 64, 8, 128, [700 + 90 * i for i in range(20)], [(0, 20, 40)]),
    ("mma_mha_h64", 8, 8, 64, [70, 90, 110, 130, 150, 33], [(0, 5, 4)]),
]


@pytest.mark.parametrize("part_blocks,prefix_part_blocks", [(16, 0), (4, 3)])
@pytest.mark.parametrize("name,N,K,H,ctx,groups", FUSED_PREFIX_CASES, ids=[c[0] for c in FUSED_PREFIX_CASES])
def test_fused_prefix_step_equals_separate_calls(pkv, oracle, name, N, K, H, ctx, groups, part_blocks,
                                                 prefix_part_blocks):
    """pkv_decode_step_prefix (the suffix pass's producers append each new row before loading its
    block) equals pkv_slot_mapping + pkv_append + pkv_decode_attn_prefix bit for bit -- out, lse,
    slots, both pools, flags -- on the mma.sync path and on both tcgen05 forms (whose suffix pass
    overlaps the prefix pass on the GPU), with an empty sequence outside every group, a member whose
    new token opens a block (ctx = 16 k + 1) and suffixes that span several partitions; and matches
    the oracle's plain decode on every row."""
    w = gen.make_workload(f"fp_{name}", 171, N, K, H, ctx)
    tables, starts, pblocks = share_prefixes(w, groups)
    q, kn, vn = bf16_dev(w.q), bf16_dev(w.k_new), bf16_dev(w.v_new)
    bt, cl = i32_dev(tables), i32_dev(w.context_lens)
    gs, pbd = i32_dev(starts), i32_dev(pblocks)
    max_group, max_prefix = int(np.max(np.diff(starts))), int(pblocks.max())
    nbytes = pkv.pkv_prefix_workspace_bytes(w.B, N, H, tables.shape[1], max_prefix, part_blocks,
                                            prefix_part_blocks)
    res = []
    for fused in (False, True):
        kc, vc = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, N), float("nan"), dtype=torch.float32, device="cuda")
        slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            pkv.check(pkv.pkv_decode_step_prefix(q, kn, vn, kc, vc, bt, cl, w.scale, gs, pbd, max_group,
                                                 max_prefix, out, lse, slots, part_blocks, ws, err,
                                                 prefix_partition_blocks=prefix_part_blocks))
        else:
            pkv.check(pkv.pkv_slot_mapping(bt, cl, w.num_blocks, slots, err))
            pkv.check(pkv.pkv_append(kn, vn, slots, kc, vc, err))
            pkv.check(pkv.pkv_decode_attn_prefix(q, kc, vc, bt, cl, w.scale, gs, pbd, max_group, max_prefix,
                                                 out, lse, part_blocks, ws, err,
                                                 prefix_partition_blocks=prefix_part_blocks))
        res.append((out, lse, slots, kc, vc, pkv.pkv_read_err_flag(err)))
    (o1, l1, s1, k1, v1, f1), (o2, l2, s2, k2, v2, f2) = res
    assert f1 == f2 == (pkv.PKV_OK, 0)
    ref_slots = oracle.slot_mapping(tables, w.context_lens)
    assert torch.equal(s1, s2) and np.array_equal(s2.cpu().numpy(), ref_slots)
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.append(w.k_new, w.v_new, ref_slots, kc, vc)
    assert np.array_equal(bf16_host(k2), kc) and np.array_equal(bf16_host(v2), vc)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    ref, ref_lse = oracle.decode(w.q, kc, vc, tables, w.context_lens, w.scale)
    assert_close(out_f64(o2), ref, f"fused prefix step {name}")
    assert_lse_close(l2.cpu().numpy().astype(np.float64), ref_lse, f"fused prefix step {name}")


def test_fused_prefix_step_refuses_a_write_into_shared_blocks(pkv, oracle):
    """A member whose context ends exactly at its group's shared blocks would append into a block
    every member reads: the fused step flags it (PKV_FLAG_GROUP_RANGE), writes no row (slot -1, both
    pools unchanged there) and still computes every other sequence as the oracle does."""
    w = gen.make_workload("fp_shared_end", 172, 32, 8, 128, [200, 96, 250, 300])
    tables, starts, pblocks = share_prefixes(w, [(0, 1, 6), (2, 4, 6)])
    # sequence 1 joins group 0 with ctx = 96 = 16 * 6: its new token would land in a shared block
    starts = np.array([0, 2, 4], dtype=np.int32)
    pblocks = np.array([6, 6], dtype=np.int32)
    tables[1, :6] = tables[0, :6]
    q, kn, vn = bf16_dev(w.q), bf16_dev(w.k_new), bf16_dev(w.v_new)
    kc, vc = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
    k_before, v_before = kc.clone(), vc.clone()
    out = torch.empty_like(q)
    slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
    ws = torch.empty(pkv.pkv_prefix_workspace_bytes(w.B, w.N, w.H, tables.shape[1], 6, 16, 0),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.check(pkv.pkv_decode_step_prefix(q, kn, vn, kc, vc, i32_dev(tables), i32_dev(w.context_lens), w.scale,
                                         i32_dev(starts), i32_dev(pblocks), 2, 6, out, None, slots, 16, ws, err))
    st, flag = pkv.pkv_read_err_flag(err)
    assert st == pkv.PKV_ERR_RANGE and flag == pkv.PKV_FLAG_GROUP_RANGE
    s = slots.cpu().numpy()
    ref_slots = oracle.slot_mapping(tables, w.context_lens)
    assert s[1] == -1 and np.array_equal(s[[0, 2, 3]], ref_slots[[0, 2, 3]])
    # only the other sequences' rows were written, in both pools
    written = sorted(int(x) for x in ref_slots[[0, 2, 3]])
    for after, before in ((kc, k_before), (vc, v_before)):
        rows = (after.view(torch.int16) != before.view(torch.int16)).any(-1).any(-1).view(-1)
        assert torch.nonzero(rows).view(-1).cpu().tolist() == written
    kh, vh = w.k_cache.copy(), w.v_cache.copy()
    keep = [0, 2, 3]
    oracle.append(w.k_new[keep], w.v_new[keep], ref_slots[keep], kh, vh)
    ref, _ = oracle.decode(w.q, kh, vh, tables, w.context_lens, w.scale)
    assert_close(out_f64(out)[keep], ref[keep], "fused prefix step, other sequences")


@pytest.mark.parametrize("kind", ["prefix_tc128", "prefix_tc32", "multi_T8"])
def test_graph_replay_of_overlapped_launches_equals_eager(pkv, oracle, kind):
    """Steps whose launches overlap on the GPU through programmatic serialization -- the tcgen05
    prefix pass with the suffix pass launched behind it and the merge behind both, and the tcgen05
    multi-token kernel with its merge behind it -- captured in a CUDA graph and replayed three times
    give bit for bit what the eager launches give (the graph keeps the programmatic dependencies),
    and match the oracle."""
    from paged_kv_decode_slot_gb300.step import MultiTokenStep, PrefixDecodeStep, StepGraph
    if kind.startswith("prefix"):
        groups = [(0, 12, 8)] if kind == "prefix_tc128" else [(0, 4, 9)]
        ctx = [130 + 7 * i for i in range(12)] if kind == "prefix_tc128" else [150, 170, 190, 210, 77]
        w = gen.make_workload(f"g_{kind}", 181, 64, 8, 128, ctx)
        tables, starts, pblocks = share_prefixes(w, groups)

        def make():
            return PrefixDecodeStep(bf16_dev(w.q), bf16_dev(w.k_new), bf16_dev(w.v_new), bf16_dev(w.k_cache),
                                    bf16_dev(w.v_cache), i32_dev(tables), i32_dev(w.context_lens), w.scale,
                                    i32_dev(starts), i32_dev(pblocks), int(np.max(np.diff(starts))),
                                    int(pblocks.max()), partition_blocks=4, prefix_partition_blocks=3)
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        oracle.append(w.k_new, w.v_new, oracle.slot_mapping(tables, w.context_lens), kc, vc)
        ref, _ = oracle.decode(w.q, kc, vc, tables, w.context_lens, w.scale)
    else:
        w = gen.make_workload("g_multi", 182, 16, 4, 128, [0, 3, 17, 300, 700, 1000])
        c = MultiCase(oracle, w, 8, 183)

        def make():
            return MultiTokenStep(bf16_dev(c.q), bf16_dev(c.k_new), bf16_dev(c.v_new), bf16_dev(w.k_cache),
                                  bf16_dev(w.v_cache), i32_dev(w.block_tables), i32_dev(w.context_lens), w.scale,
                                  partition_blocks=8)
        ref, _ = c.reference(oracle)
    eager = make()
    assert eager.launches_per_step() >= 2
    eager.run()
    graphed = make()
    g = StepGraph(graphed)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.out.view(torch.int16), graphed.out.view(torch.int16)), kind
    assert torch.equal(eager.lse, graphed.lse) and torch.equal(eager.slot_mapping, graphed.slot_mapping)
    assert torch.equal(eager.k_cache.view(torch.int16), graphed.k_cache.view(torch.int16))
    assert_close(out_f64(graphed.out), ref, f"graph replay {kind}")


def test_fused_prefix_step_bad_block_is_flagged_and_skipped(pkv, oracle):
    """A table entry outside the pool in the block that holds a sequence's new token (past the
    shared prefix): the fused shared-prefix step flags it, writes nothing there and reports slot -1,
    as pkv_slot_mapping + pkv_append do, and computes every other sequence as the oracle does."""
    w = gen.make_workload("fp_bad", 184, 64, 8, 128, [150, 170, 190, 210, 77])
    tables, starts, pblocks = share_prefixes(w, [(0, 4, 9)])
    tables = tables.copy()
    tables[2, (int(w.context_lens[2]) - 1) // 16] = w.num_blocks + 3
    q, kn, vn = bf16_dev(w.q), bf16_dev(w.k_new), bf16_dev(w.v_new)
    bt, cl = i32_dev(tables), i32_dev(w.context_lens)
    res = []
    for fused in (False, True):
        kc, vc = bf16_dev(w.k_cache), bf16_dev(w.v_cache)
        out = torch.empty_like(q)
        slots = torch.full((w.B,), -7, dtype=torch.int64, device="cuda")
        ws = torch.empty(pkv.pkv_prefix_workspace_bytes(w.B, w.N, w.H, tables.shape[1], 9, 4, 0),
                         dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            pkv.check(pkv.pkv_decode_step_prefix(q, kn, vn, kc, vc, bt, cl, w.scale, i32_dev(starts), i32_dev(pblocks),
                                                 4, 9, out, None, slots, 4, ws, err))
        else:
            pkv.check(pkv.pkv_slot_mapping(bt, cl, w.num_blocks, slots, err))
            pkv.check(pkv.pkv_append(kn, vn, slots, kc, vc, err))
            pkv.check(pkv.pkv_decode_attn_prefix(q, kc, vc, bt, cl, w.scale, i32_dev(starts), i32_dev(pblocks), 4, 9,
                                                 out, None, 4, ws, err))
        res.append((out, slots, kc, vc, pkv.pkv_read_err_flag(err)))
    (o1, s1, k1, v1, f1), (o2, s2, k2, v2, f2) = res
    assert f1 == f2 and f2[1] & pkv.PKV_FLAG_BLOCK_RANGE
    assert torch.equal(s1, s2) and int(s2[2]) == -1
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16)) and torch.equal(v1.view(torch.int16),
                                                                                   v2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    kh, vh = w.k_cache.copy(), w.v_cache.copy()
    keep = [0, 1, 3, 4]
    oracle.append(w.k_new[keep], w.v_new[keep], oracle.slot_mapping(tables, w.context_lens)[keep], kh, vh)
    ref, _ = oracle.decode(w.q, kh, vh, tables, w.context_lens, w.scale)
    assert_close(out_f64(o2)[keep], ref[keep], "fused prefix step with a bad block, other sequences")
