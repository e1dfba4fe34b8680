"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle, check):
    check(oracle)


def test_allocated_cache_bytes_match_formula(oracle):
    # a pool of num_blocks blocks of 16 tokens holds 2 * num_blocks*16 * K * H * 2 bytes of K and V
    from paged_kv_decode_slot_gb300 import inputs as gen
    w = gen.make_config("tiny")
    allocated = w.k_cache.nbytes + w.v_cache.nbytes
    assert allocated == oracle.kv_bytes(1, w.K, w.H, w.num_blocks * 16, 2)
