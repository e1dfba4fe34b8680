"""Expiring in-kernel waits on the GPU: no fault, no hang, the context stays usable.

Every wait inside the kernels is bounded (pkv_set_wait_limit_ns, default 2 s).  An expired wait
sets PKV_FLAG_TIMEOUT; the kernel stops issuing, drains the copies it started, releases what it
holds (tensor memory included) and returns, and the unit's result is void.
  * pkv_check_wait_expiry waits, with the same bounded wait, on an mbarrier nothing completes:
    the expiry is certain and flagged.
  * Every attention path runs with pkv_debug_withhold_tile(3) and a 1 ms limit: each CTA's
    producer skips its fourth tile (no load, no barrier arrival -- a flag nothing sets), so the
    consumer's wait on it expires and every CTA with four or more tiles takes its abort path
    (stop issuing, drain the copies it started, let its MMAs finish, release its tensor memory,
    count toward the merge, return).  Only PKV_FLAG_TIMEOUT may be flagged, and it must be.
    The same step then runs again with the defaults and must match the oracle: the context
    works, the fused append lands, and the split workspace's merge counters are back at zero.
    The hook exists only in a test build of the library (-DPKV_TEST_HOOKS, built here next to
    the product library); each of these cases runs in a child process that loads that build
    through PKV_LIBRARY, so the product library the other tests load carries no hook.
"""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for _p in (ROOT, HERE):
    if _p not in sys.path:
        sys.path.insert(0, _p)

from devutil import assert_close, bf16_dev, i32_dev, out_f64, upload  # noqa: E402
from paged_kv_decode_slot_gb300 import inputs as gen  # noqa: E402

pytestmark = pytest.mark.gpu

HOOKS_DIR = os.path.join(ROOT, "_build", "test_hooks")
HOOKS_LIB = os.path.join(HOOKS_DIR, "libpagedkv_test_hooks.so")
KINDS = ["single", "split", "split_fp8", "multi_tc", "multi_mma", "prefix"]


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_slot_gb300.build import build_library
    build_library()
    import paged_kv_decode_slot_gb300 as pkv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkv


def test_wait_that_never_completes_expires_and_is_flagged(pkv):
    prev = pkv.pkv_set_wait_limit_ns(1_000_000)  # 1 ms
    try:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.check(pkv.pkv_check_wait_expiry(err))
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_wait_limit_ns(prev)
    st, flag = pkv.pkv_read_err_flag(err)
    assert flag == pkv.PKV_FLAG_TIMEOUT and st != pkv.PKV_OK
    # the context is fine afterwards
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2


def _flags_with_withheld_tile(pkv, run):
    """Run `run(err)` with tile 3 of every CTA withheld and a 1 ms wait limit; return the flags."""
    prev = pkv.pkv_set_wait_limit_ns(1_000_000)
    prev_w = pkv.pkv_debug_withhold_tile(3)
    try:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        run(err)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_debug_withhold_tile(prev_w)
        pkv.pkv_set_wait_limit_ns(prev)
    assert prev_w == -1
    _, flag = pkv.pkv_read_err_flag(err)
    assert flag == pkv.PKV_FLAG_TIMEOUT, f"expected exactly the timeout flag, got {flag:#x}"
    return flag


@pytest.fixture(scope="module")
def hooks_lib():
    from paged_kv_decode_slot_gb300.build import build_library
    return build_library(out=HOOKS_LIB, defines=("PKV_TEST_HOOKS",), build_dir=HOOKS_DIR)


@pytest.mark.parametrize("kind", KINDS)
def test_kernels_survive_expired_waits_and_recover(hooks_lib, kind):
    env = dict(os.environ, PKV_LIBRARY=hooks_lib)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), kind], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "RECOVERED" in r.stdout, (r.stdout[-4000:], r.stderr[-4000:])


def expired_waits_case(kind: str) -> None:
    """One case, in a process whose library is the test build (PKV_LIBRARY)."""
    import oracle as oracle_mod
    import paged_kv_decode_slot_gb300 as pkv
    from paged_kv_decode_slot_gb300.step import (AttentionPlan, DecodeStep, DecodeStepFp8, MultiTokenStep,
                                                 PrefixDecodeStep, plan_attention)
    assert pkv.binding.HAS_TEST_HOOKS, "the child must load the -DPKV_TEST_HOOKS build"
    oracle = oracle_mod.default()
    w = gen.make_config("l3_8b_b16")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if kind in ("single", "split"):
        plan = AttentionPlan("single") if kind == "single" else plan_attention(w.B, w.K, w.max_blocks, sms)

        def make(err):
            d = upload(w)
            return DecodeStep(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                              d["context_lens"], w.scale, plan=plan, err_flag=err)
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        oracle.append(w.k_new, w.v_new, oracle.slot_mapping(w.block_tables, w.context_lens), kc, vc)
        ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    elif kind == "split_fp8":
        ks = np.full(w.K, 0.02, dtype=np.float32)
        vs = np.full(w.K, 0.02, dtype=np.float32)
        kc8, vc8 = oracle.quantize_fp8(w.k_cache, ks), oracle.quantize_fp8(w.v_cache, vs)

        def make(err):
            return DecodeStepFp8(bf16_dev(w.q), bf16_dev(w.k_new), bf16_dev(w.v_new),
                                 torch.from_numpy(kc8).cuda(), torch.from_numpy(vc8).cuda(),
                                 torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(),
                                 i32_dev(w.block_tables), i32_dev(w.context_lens), w.scale, err_flag=err)
        kc8a, vc8a = kc8.copy(), vc8.copy()
        oracle.append_fp8(w.k_new, w.v_new, ks, vs, oracle.slot_mapping(w.block_tables, w.context_lens), kc8a, vc8a)
        ref, _ = oracle.decode_fp8(w.q, kc8a, vc8a, ks, vs, w.block_tables, w.context_lens, w.scale)
    elif kind in ("multi_tc", "multi_mma"):
        T = 8 if kind == "multi_tc" else 2
        qm = gen.normal_bf16(7, 1, (w.B, T, w.N, w.H))
        knm = gen.normal_bf16(7, 2, (w.B, T, w.K, w.H))
        vnm = gen.normal_bf16(7, 3, (w.B, T, w.K, w.H))

        def make(err):
            return MultiTokenStep(bf16_dev(qm), bf16_dev(knm), bf16_dev(vnm), bf16_dev(w.k_cache),
                                  bf16_dev(w.v_cache), i32_dev(w.block_tables), i32_dev(w.context_lens), w.scale,
                                  err_flag=err)
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        slots = oracle.slot_mapping_multi(w.block_tables, w.context_lens, T)
        oracle.append(knm.reshape(-1, w.K, w.H), vnm.reshape(-1, w.K, w.H), slots.reshape(-1), kc, vc)
        ref, _ = oracle.decode_multi(qm, kc, vc, w.block_tables, w.context_lens, w.scale)
    else:
        w = gen.make_config("prefix_l3_70b")
        gs, pb = w.prefix_groups()

        def make(err):
            d = upload(w)
            return PrefixDecodeStep(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], w.scale, i32_dev(gs), i32_dev(pb), int(np.max(np.diff(gs))),
                                    int(pb.max()), partition_blocks=16, err_flag=err)
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        oracle.append(w.k_new, w.v_new, oracle.slot_mapping(w.block_tables, w.context_lens), kc, vc)
        ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)

    err0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = make(err0)
    _flags_with_withheld_tile(pkv, lambda err: (setattr(step, "err_flag", err), step.run()))
    # the same step object (its workspace and counters included) with the default limit
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step.err_flag = err
    step.run()
    torch.cuda.synchronize()
    assert pkv.pkv_read_err_flag(err) == (pkv.PKV_OK, 0)
    assert_close(out_f64(step.out), ref, f"{kind} after expired waits")


if __name__ == "__main__":
    expired_waits_case(sys.argv[1])
    print("RECOVERED", flush=True)
