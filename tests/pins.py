"""Pins for the oracle: checks against facts the pages and mathematics fix.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with something other than itself: a value the pages
print, a library routine (torch's scaled_dot_product_attention, mpmath at
40 digits), a closed form, an invariant, or brute force on tiny inputs.
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on deliberately broken copies of it and expects a failure each.
"""
from __future__ import annotations

import math
import os

import numpy as np

from paged_kv_decode_slot_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BS = 16


def read_kv_bytes_golden():
    rows = []
    with open(os.path.join(GOLDEN, "kv_bytes.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            nums, cite = line.split("|", 1)
            vals = [int(x) for x in nums.split()]
            rows.append((vals[:5], vals[5], cite.strip()))
    return rows


def to_f64(bits):
    return gen.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def paged_from_contiguous(k_seqs, v_seqs, seed, extra_blocks=3, spare_cols=1):
    """Scatter per-sequence contiguous K/V ([ctx_b, K, H] uint16) into a shuffled paged pool.

    The construction goes contiguous -> paged; the oracle goes paged -> contiguous.
    Unused slots are NaN so that a stray read shows.
    """
    K, H = k_seqs[0].shape[1], k_seqs[0].shape[2]
    ctx = np.array([k.shape[0] for k in k_seqs], dtype=np.int32)
    nb = [(c + BS - 1) // BS for c in ctx.tolist()]
    total = sum(nb) + extra_blocks
    perm = np.random.default_rng(seed).permutation(total)
    kc = np.full((total, BS, K, H), gen.BF16_NAN, dtype=np.uint16)
    vc = np.full((total, BS, K, H), gen.BF16_NAN, dtype=np.uint16)
    tables = np.full((len(k_seqs), max(nb) + spare_cols), -1, dtype=np.int32)
    pos = 0
    for b, (ks, vs) in enumerate(zip(k_seqs, v_seqs)):
        blocks = perm[pos:pos + nb[b]]
        pos += nb[b]
        tables[b, :nb[b]] = blocks
        t = np.arange(ks.shape[0])
        kc[blocks[t // BS], t % BS] = ks
        vc[blocks[t // BS], t % BS] = vs
    return kc, vc, tables, ctx


def random_case(seed, N, K, H, ctxs, k_mult=1.0):
    q = gen.normal_bf16(seed, 100, (len(ctxs), N, H))
    ks = [gen.normal_bf16(seed, 200 + b, (c, K, H), mult=k_mult) for b, c in enumerate(ctxs)]
    vs = [gen.normal_bf16(seed, 300 + b, (c, K, H)) for b, c in enumerate(ctxs)]
    return q, ks, vs


def sdpa_reference(q, ks, vs, scale):
    """torch scaled_dot_product_attention in float64 on contiguous K/V, per sequence."""
    import torch
    B, N, H = q.shape
    K = ks[0].shape[1]
    G = N // K
    out = np.zeros((B, N, H))
    lse = np.zeros((B, N))
    for b in range(B):
        qt = torch.from_numpy(to_f64(q[b])).reshape(1, N, 1, H)
        kt = torch.from_numpy(to_f64(ks[b])).permute(1, 0, 2).unsqueeze(0)   # [1, K, ctx, H]
        vt = torch.from_numpy(to_f64(vs[b])).permute(1, 0, 2).unsqueeze(0)
        kt = kt.repeat_interleave(G, dim=1)                                  # query group n -> n // G
        vt = vt.repeat_interleave(G, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        out[b] = o.reshape(N, H).numpy()
        s = torch.matmul(qt, kt.transpose(-1, -2)) * scale                  # [1, N, 1, ctx]
        lse[b] = torch.logsumexp(s, dim=-1).reshape(N).numpy()
    return out, lse


# ----------------------------------------------------------------------------------------
def check_kv_bytes_golden(orc):
    for (L, K, H, S, nbytes), expected, cite in read_kv_bytes_golden():
        got = orc.kv_bytes(L, K, H, S, nbytes)
        assert got == expected, f"{cite}: {got} != {expected}"


def check_paged_equals_contiguous(orc):
    cases = [(8, 2, 64, [1, 17, 64, 200], 11), (4, 4, 64, [15, 16, 33], 12),
             (8, 1, 64, [5, 48], 13), (16, 2, 128, [31, 70], 14)]
    for N, K, H, ctxs, seed in cases:
        q, ks, vs = random_case(seed, N, K, H, ctxs)
        kc, vc, tables, ctx = paged_from_contiguous(ks, vs, seed)
        scale = 1.0 / math.sqrt(H)
        out, lse = orc.decode(q, kc, vc, tables, ctx, scale)
        ref_out, ref_lse = sdpa_reference(q, ks, vs, scale)
        assert np.all(np.isfinite(out)), "oracle read a poisoned slot"
        assert np.max(np.abs(out - ref_out)) < 1e-12, (N, K, H, ctxs)
        assert np.max(np.abs(lse - ref_lse)) < 1e-12, (N, K, H, ctxs)


def check_block_permutation_invariance(orc):
    q, ks, vs = random_case(21, 8, 2, 64, [40, 97, 16])
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 1)
    out1, lse1 = orc.decode(q, kc, vc, tables, ctx, 0.125)
    # move every physical block to a new id and rewrite the tables accordingly
    perm = np.random.default_rng(5).permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    out2, lse2 = orc.decode(q, kc2, vc2, t2, ctx, 0.125)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def check_ctx1_returns_v(orc):
    q, ks, vs = random_case(31, 8, 2, 64, [1, 1, 1])
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 2)
    out, lse = orc.decode(q, kc, vc, tables, ctx, 0.125)
    G = 4
    for b in range(3):
        for n in range(8):
            assert np.array_equal(out[b, n], to_f64(vs[b][0, n // G])), (b, n)
            s = 0.125 * float(np.dot(to_f64(q[b, n]), to_f64(ks[b][0, n // G])))
            assert abs(lse[b, n] - s) <= 1e-12 * max(1.0, abs(s))


def check_constant_v(orc):
    q, ks, vs = random_case(41, 8, 2, 64, [3, 50, 129])
    c = gen.f32_to_bf16_bits(np.array([0.6875], dtype=np.float32))[0]
    vs = [np.full_like(v, c) for v in vs]
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 3)
    out, _ = orc.decode(q, kc, vc, tables, ctx, 0.125)
    assert np.max(np.abs(out - 0.6875)) < 1e-13


def check_zero_query_is_uniform_mean(orc):
    q, ks, vs = random_case(51, 8, 2, 64, [7, 33, 100])
    q = np.zeros_like(q)
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 4)
    out, lse = orc.decode(q, kc, vc, tables, ctx, 0.125)
    for b, c in enumerate(ctx.tolist()):
        mean = to_f64(vs[b]).mean(axis=0)               # [K, H]
        for n in range(8):
            assert np.max(np.abs(out[b, n] - mean[n // 4])) < 1e-13
            assert abs(lse[b, n] - math.log(c)) < 1e-13


def check_brute_force_mpmath(orc, large_logits=False):
    import mpmath
    mpmath.mp.dps = 40
    k_mult = 1024.0 if large_logits else 1.0
    q, ks, vs = random_case(61 + int(large_logits), 4, 2, 64, [9, 23, 40], k_mult=k_mult)
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 5)
    out, lse = orc.decode(q, kc, vc, tables, ctx, 0.125)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    for b in range(3):
        kf, vf = to_f64(ks[b]), to_f64(vs[b])
        for n in range(4):
            qf = to_f64(q[b, n])
            kvh = n // 2
            w = [mpmath.exp(mpmath.mpf(0.125) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(x))
                                                           for a, x in zip(qf, kf[t, kvh])))
                 for t in range(kf.shape[0])]
            z = mpmath.fsum(w)
            for h in range(0, 64, 7):
                ref = mpmath.fsum(wt * mpmath.mpf(float(vf[t, kvh, h])) for t, wt in enumerate(w)) / z
                assert abs(out[b, n, h] - float(ref)) < 1e-12, (b, n, h)
            assert abs(lse[b, n] - float(mpmath.log(z))) < 1e-9 * max(1.0, abs(float(mpmath.log(z))))


def check_large_logits(orc):
    check_brute_force_mpmath(orc, large_logits=True)


def check_partitions_merge_to_unsplit(orc):
    q, ks, vs = random_case(71, 8, 2, 64, [1, 64, 65, 150])
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 6)
    out, lse = orc.decode(q, kc, vc, tables, ctx, 0.125)
    for pt, P in ((64, 3), (16, 10), (48, 5)):       # includes empty trailing partitions
        po, pl = orc.decode_partitions(q, kc, vc, tables, ctx, 0.125, pt, P)
        assert np.all(pl[0, :, 1:] == -np.inf) and np.all(po[0, :, 1:] == 0.0)
        mo, ml = orc.lse_merge(po, pl)
        assert np.max(np.abs(mo - out)) < 1e-12 and np.max(np.abs(ml - lse)) < 1e-12
    # one partition per token: the merge is the softmax over singletons (scipy's softmax)
    from scipy.special import softmax
    po, pl = orc.decode_partitions(q, kc, vc, tables, ctx, 0.125, 1, 150)
    b, n = 3, 5
    w = softmax(pl[b, n, :ctx[b]])
    ref = (w[:, None] * to_f64(vs[b][:, n // 4])).sum(axis=0)
    mo, _ = orc.lse_merge(po, pl)
    assert np.max(np.abs(mo[b, n] - ref)) < 1e-12


def check_ctx0(orc):
    q, ks, vs = random_case(81, 4, 2, 64, [5, 9])
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 7)
    ctx = ctx.copy()
    ctx[0] = 0
    out, lse = orc.decode(q, kc, vc, tables, ctx, 0.125)
    assert np.all(out[0] == 0.0) and np.all(lse[0] == -np.inf)


def check_slot_mapping(orc):
    # identity tables: sequence b owns blocks b*M .. b*M+M-1 in order, so slot = b*M*16 + ctx-1
    M = 5
    ctx = np.array([1, 16, 17, 80, 33], dtype=np.int32)
    tables = (np.arange(5)[:, None] * M + np.arange(M)[None, :]).astype(np.int32)
    slots = orc.slot_mapping(tables, ctx)
    assert np.array_equal(slots, np.arange(5) * M * 16 + ctx - 1)
    # shuffled tables: the newest token's block is the table entry of block (ctx-1)//16
    rng = np.random.default_rng(3)
    tables = rng.permutation(40).reshape(5, 8).astype(np.int32)
    ctx = np.array([1, 16, 17, 100, 127], dtype=np.int32)
    slots = orc.slot_mapping(tables, ctx)
    for b in range(5):
        p = int(ctx[b]) - 1
        blk = int(tables[b, p // 16])
        assert slots[b] == blk * 16 + p % 16
        # and its K row lies inside that block's byte range of the [nb, 16, K, H] pool
        assert blk * 16 <= slots[b] < blk * 16 + 16
    assert orc.slot_mapping(tables[:1], np.array([0], dtype=np.int32))[0] == -1


def check_append_gather_roundtrip(orc):
    w = gen.make_config("tiny")
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    slots = orc.slot_mapping(w.block_tables, w.context_lens)
    orc.append(w.k_new, w.v_new, slots, kc, vc)
    # exactly the new rows changed, byte for byte
    changed = np.zeros(kc.shape[:2], dtype=bool)
    for s in slots.tolist():
        changed[s // 16, s % 16] = True
    assert np.array_equal(kc[~changed].view(np.uint16), w.k_cache[~changed].view(np.uint16))
    ko, vo, cu = orc.gather(kc, vc, w.block_tables, w.context_lens)
    for b in range(w.B):
        last = int(cu[b + 1]) - 1                     # position ctx-1 of sequence b
        assert np.array_equal(ko[last], w.k_new[b]) and np.array_equal(vo[last], w.v_new[b])
    # a skipped (negative) slot leaves the cache untouched
    kc2, vc2 = w.k_cache.copy(), w.v_cache.copy()
    orc.append(w.k_new, w.v_new, np.full(w.B, -1, dtype=np.int64), kc2, vc2)
    assert np.array_equal(kc2, w.k_cache) and np.array_equal(vc2, w.v_cache)


def check_gather_inverts_scatter(orc):
    q, ks, vs = random_case(91, 8, 2, 64, [3, 16, 17, 45])
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 8)
    ko, vo, cu = orc.gather(kc, vc, tables, ctx)
    assert np.array_equal(ko, np.concatenate(ks)) and np.array_equal(vo, np.concatenate(vs))


# ---------------------------------------- FP8 -------------------------------------------
def check_e4m3_decode_table(orc):
    """Values the E4M3 format definition fixes (OCP 8-bit floating point, E4M3)."""
    t = orc.e4m3_decode_table()
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0x80: -0.0,
             0xB8: -1.0, 0xFE: -448.0}
    for c, v in fixed.items():
        assert t[c] == v and np.signbit(t[c]) == np.signbit(v), (hex(c), t[c], v)
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    finite = t[np.isfinite(t)]
    assert finite.size == 254 and len(set(finite[finite > 0].tolist())) == 126


def check_e4m3_encode_nearest_even(orc):
    """Brute force: the code of x is the nearest finite e4m3 value, ties to the even code."""
    t = orc.e4m3_decode_table()
    codes = [c for c in range(256) if np.isfinite(t[c])]
    rng = np.random.default_rng(9)
    xs = np.concatenate([rng.normal(0, 1, 400), rng.normal(0, 100, 200), rng.uniform(-520, 520, 200),
                         [464.0, -470.0, 479.9, 1000.0, -1e30],                # beyond the largest code
                         rng.uniform(-2.0 ** -6, 2.0 ** -6, 200),
                         [(t[c] + t[c + 1]) / 2 for c in range(0x00, 0x7D)]])   # exact midpoints
    for x in xs.astype(np.float32):
        got = orc.e4m3_encode(float(x))
        if abs(x) >= 448:
            assert t[got] == np.copysign(448.0, x), (x, hex(got))
            continue
        d = [abs(t[c] - float(x)) for c in codes]
        best = min(d)
        cands = [c for c, dc in zip(codes, d) if dc == best]
        if len(cands) > 1:                       # a tie: the even code (zero: keep the sign)
            cands = [c for c in cands if c & 1 == 0] or cands
            if float(x) == 0.0:
                cands = [0x80 if np.signbit(x) else 0x00]
        assert got in cands, (float(x), hex(got), [hex(c) for c in cands])
    for c in codes:                              # representable values encode to themselves
        assert t[orc.e4m3_encode(float(t[c]))] == t[c]


def check_fp8_attention_is_dequantized_attention(orc):
    """decode_fp8 == the bf16-path oracle's definition on the dequantized K/V (torch SDPA)."""
    q, ks, vs = random_case(95, 8, 2, 128, [1, 17, 70])
    k_scale = np.array([0.011, 0.013], dtype=np.float32)     # 448 * scale > every |value| here
    v_scale = np.array([0.013, 0.0125], dtype=np.float32)
    k8 = [orc.quantize_fp8(k, k_scale) for k in ks]
    v8 = [orc.quantize_fp8(v, v_scale) for v in vs]
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 10)
    kc8 = orc.quantize_fp8(kc, k_scale)
    vc8 = orc.quantize_fp8(vc, v_scale)
    out, lse = orc.decode_fp8(q, kc8, vc8, k_scale, v_scale, tables, ctx, 1 / math.sqrt(128))
    t = orc.e4m3_decode_table()
    import torch
    for b in range(3):
        kd = (t[k8[b]] * k_scale[None, :, None]).astype(np.float64)      # [ctx, K, H]
        vd = (t[v8[b]] * v_scale[None, :, None]).astype(np.float64)
        qt = torch.from_numpy(to_f64(q[b])).reshape(1, 8, 1, 128)
        kt = torch.from_numpy(kd).permute(1, 0, 2).unsqueeze(0).repeat_interleave(4, dim=1)
        vt = torch.from_numpy(vd).permute(1, 0, 2).unsqueeze(0).repeat_interleave(4, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=1 / math.sqrt(128))
        assert np.max(np.abs(out[b] - ref.reshape(8, 128).numpy())) < 1e-12
    # context 1: the output is that token's dequantized V, within e4m3 rounding of the bf16 V
    # (half a unit of the 3-bit mantissa: 2^-4 relative, or half the subnormal step 2^-10 * scale)
    v0 = to_f64(vs[0][0])                                        # [K, H]
    for n in range(8):
        kvh = n // 4
        bound = np.maximum(np.abs(v0[kvh]) * 2.0 ** -4, 2.0 ** -10 * float(v_scale[kvh])) * (1 + 1e-6)
        assert np.all(np.abs(out[0, n] - v0[kvh]) <= bound)


def check_fp8_block_scales(orc):
    """Per-(physical block, KV head) scales [num_blocks, K]: (1) quantizing a pool equals
    quantizing each block with the per-head scales of that block; (2) attention equals SDPA on
    the values dequantized with the scales of each token's physical block (the tables are
    permuted, so a logical block index would pick other scales); (3) an append quantizes the new
    row with the scales of the block its slot lies in."""
    q, ks, vs = random_case(97, 8, 2, 128, [5, 17, 70])
    kc, vc, tables, ctx = paged_from_contiguous(ks, vs, 12)
    nblk = kc.shape[0]
    rng = np.random.default_rng(97)
    k_sc = rng.uniform(0.004, 0.02, size=(nblk, 2)).astype(np.float32)
    v_sc = rng.uniform(0.004, 0.02, size=(nblk, 2)).astype(np.float32)
    kc8 = orc.quantize_fp8(kc, k_sc)
    vc8 = orc.quantize_fp8(vc, v_sc)
    for blk in range(nblk):
        assert np.array_equal(kc8[blk], orc.quantize_fp8(kc[blk], k_sc[blk]))
        assert np.array_equal(vc8[blk], orc.quantize_fp8(vc[blk], v_sc[blk]))
    out, lse = orc.decode_fp8(q, kc8, vc8, k_sc, v_sc, tables, ctx, 1 / math.sqrt(128))
    t = orc.e4m3_decode_table()
    import torch
    for b in range(3):
        n = int(ctx[b])
        blocks = tables[b, np.arange(n) // BS]
        offs = np.arange(n) % BS
        kd = t[kc8[blocks, offs]] * k_sc[blocks][:, :, None].astype(np.float64)   # [n, K, H]
        vd = t[vc8[blocks, offs]] * v_sc[blocks][:, :, None].astype(np.float64)
        qt = torch.from_numpy(to_f64(q[b])).reshape(1, 8, 1, 128)
        kt = torch.from_numpy(kd).permute(1, 0, 2).unsqueeze(0).repeat_interleave(4, dim=1)
        vt = torch.from_numpy(vd).permute(1, 0, 2).unsqueeze(0).repeat_interleave(4, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=1 / math.sqrt(128))
        assert np.max(np.abs(out[b] - ref.reshape(8, 128).numpy())) < 1e-12
    kn = gen.normal_bf16(97, 400, (3, 2, 128))
    vn = gen.normal_bf16(97, 401, (3, 2, 128))
    slots = np.array([tables[0, 0] * BS + 5, tables[2, 4] * BS + 15, tables[1, 1] * BS + 2], dtype=np.int64)
    orc.append_fp8(kn, vn, k_sc, v_sc, slots, kc8, vc8)
    for i, s_ in enumerate(slots.tolist()):
        blk = s_ // BS
        assert np.array_equal(kc8[blk, s_ % BS], orc.quantize_fp8(kn[i:i + 1], k_sc[blk])[0])
        assert np.array_equal(vc8[blk, s_ % BS], orc.quantize_fp8(vn[i:i + 1], v_sc[blk])[0])


def check_fp8_append_roundtrip(orc):
    w = gen.make_config("tiny")
    k_scale = np.array([0.01, 0.02], dtype=np.float32)
    v_scale = np.array([0.015, 0.005], dtype=np.float32)
    kc8 = orc.quantize_fp8(w.k_cache, k_scale)
    vc8 = orc.quantize_fp8(w.v_cache, v_scale)
    slots = orc.slot_mapping(w.block_tables, w.context_lens)
    before_k = kc8.copy()
    orc.append_fp8(w.k_new, w.v_new, k_scale, v_scale, slots, kc8, vc8)
    for b, s_ in enumerate(slots.tolist()):
        assert np.array_equal(kc8[s_ // 16, s_ % 16], orc.quantize_fp8(w.k_new[b:b + 1], k_scale)[0])
        assert np.array_equal(vc8[s_ // 16, s_ % 16], orc.quantize_fp8(w.v_new[b:b + 1], v_scale)[0])
    changed = np.any(kc8 != before_k, axis=(2, 3))
    assert sorted(map(tuple, np.argwhere(changed))) == sorted((s_ // 16, s_ % 16) for s_ in slots.tolist())


# ------------------------------- several query tokens ------------------------------------
def masked_sdpa_reference(q, ks, vs, scale):
    """torch SDPA (float64) with an explicit boolean mask: the T query rows of a sequence of
    ctx keys are its last T positions; row t may see keys 0 .. ctx - T + t."""
    import torch
    B, T, N, H = q.shape
    K = ks[0].shape[1]
    G = N // K
    out = np.zeros((B, T, N, H))
    for b in range(B):
        ctx = ks[b].shape[0]
        qt = torch.from_numpy(to_f64(q[b])).permute(1, 0, 2).unsqueeze(0)   # [1, N, T, H]
        kt = torch.from_numpy(to_f64(ks[b])).permute(1, 0, 2).unsqueeze(0).repeat_interleave(G, dim=1)
        vt = torch.from_numpy(to_f64(vs[b])).permute(1, 0, 2).unsqueeze(0).repeat_interleave(G, dim=1)
        rows = torch.arange(T).unsqueeze(1) + (ctx - T)
        mask = torch.arange(ctx).unsqueeze(0) <= rows                        # [T, ctx]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        out[b] = o[0].permute(1, 0, 2).numpy()
    return out


def check_multi_query_equals_masked_sdpa(orc):
    for N, K, H, ctxs, T, seed in [(8, 2, 64, [4, 17, 40], 4, 21), (16, 2, 128, [2, 33], 2, 22),
                                   (4, 4, 64, [16, 31], 3, 23)]:
        _, ks, vs = random_case(seed, N, K, H, ctxs)
        q = gen.normal_bf16(seed, 400, (len(ctxs), T, N, H))
        kc, vc, tables, ctx = paged_from_contiguous(ks, vs, seed)
        scale = 1.0 / math.sqrt(H)
        out, lse = orc.decode_multi(q, kc, vc, tables, ctx, scale)
        ref = masked_sdpa_reference(q, ks, vs, scale)
        assert np.all(np.isfinite(out))
        assert np.max(np.abs(out - ref)) < 1e-12, (N, K, H, ctxs, T)


def check_multi_query_is_a_sequence_of_decode_steps(orc):
    """Verifying T tokens at once gives, for token t, exactly what a one-token decode step at
    its position gives (the context cut after that token)."""
    w = gen.make_workload("pin_multi", 24, 8, 2, 64, [5, 16, 17, 50])
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    T = 4
    slots = orc.slot_mapping_multi(w.block_tables, w.context_lens, T)
    new_k = gen.normal_bf16(24, 500, (w.B, T, w.K, w.H))
    new_v = gen.normal_bf16(24, 501, (w.B, T, w.K, w.H))
    orc.append(new_k.reshape(-1, w.K, w.H), new_v.reshape(-1, w.K, w.H), slots.reshape(-1), kc, vc)
    q = gen.normal_bf16(24, 502, (w.B, T, w.N, w.H))
    out, lse = orc.decode_multi(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    for t in range(T):
        cut = np.maximum(w.context_lens - T + t + 1, 0).astype(np.int32)
        o1, l1 = orc.decode(q[:, t], kc, vc, w.block_tables, cut, w.scale)
        assert np.array_equal(out[:, t], o1) and np.array_equal(lse[:, t], l1), t


def check_slot_mapping_multi(orc):
    B, T, max_nb = 3, 5, 4
    tables = np.arange(B * max_nb, dtype=np.int32).reshape(B, max_nb)[:, ::-1].copy()
    ctx = np.array([3, 16, 40], dtype=np.int32)
    got = orc.slot_mapping_multi(tables, ctx, T)
    for b in range(B):
        for t in range(T):
            pos = int(ctx[b]) - T + t
            want = -1 if pos < 0 else int(tables[b, pos // BS]) * BS + pos % BS
            assert got[b, t] == want, (b, t, got[b, t], want)


def check_copy_blocks(orc):
    """The copy equals numpy's; a sequence whose shared partial block is replaced by a private
    copy (copy-on-write) attends exactly as before."""
    w = gen.make_workload("pin_cow", 25, 8, 2, 64, [20, 40, 9], pool_blocks=10)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    ref_k, ref_v = kc.copy(), vc.copy()
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = [x for x in range(w.num_blocks) if x not in used]
    pairs = np.array([[w.block_tables[0, 1], free[0]], [w.block_tables[1, 2], free[1]]], dtype=np.int32)
    orc.copy_blocks(kc, vc, pairs)
    for src, dst in pairs:
        ref_k[dst] = ref_k[src]
        ref_v[dst] = ref_v[src]
    assert np.array_equal(kc.view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(vc.view(np.uint16), ref_v.view(np.uint16))
    before, lse_b = orc.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    tables = w.block_tables.copy()
    tables[0, 1], tables[1, 2] = pairs[0, 1], pairs[1, 1]
    after, lse_a = orc.decode(w.q, kc, vc, tables, w.context_lens, w.scale)
    assert np.array_equal(np.nan_to_num(before, nan=7.0), np.nan_to_num(after, nan=7.0))


ALL_CHECKS = [check_kv_bytes_golden, check_paged_equals_contiguous,
              check_block_permutation_invariance, check_ctx1_returns_v, check_constant_v,
              check_zero_query_is_uniform_mean, check_brute_force_mpmath, check_large_logits,
              check_partitions_merge_to_unsplit, check_ctx0, check_slot_mapping,
              check_append_gather_roundtrip, check_gather_inverts_scatter,
              check_e4m3_decode_table, check_e4m3_encode_nearest_even,
              check_fp8_attention_is_dequantized_attention, check_fp8_block_scales, check_fp8_append_roundtrip,
              check_multi_query_equals_masked_sdpa, check_multi_query_is_a_sequence_of_decode_steps,
              check_slot_mapping_multi, check_copy_blocks]
