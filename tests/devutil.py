"""Helpers for the GPU tests: upload seeded workloads, compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_decode_slot_gb300 import inputs as gen

# Attention output tolerance against the float64 oracle (bf16 inputs and output, fp32
# accumulation): maximum absolute error 2e-2 and mean absolute error 2e-3 per case.
MAX_ABS_TOL = 2e-2
MEAN_ABS_TOL = 2e-3
# lse is an fp32 quantity (running max plus log of an fp32 sum of bf16-rounded weights).
LSE_ABS_TOL = 2e-2


def bf16_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def upload(w: gen.Workload, device="cuda") -> dict:
    return dict(q=bf16_dev(w.q, device), k_cache=bf16_dev(w.k_cache, device),
                v_cache=bf16_dev(w.v_cache, device), k_new=bf16_dev(w.k_new, device),
                v_new=bf16_dev(w.v_new, device), block_tables=i32_dev(w.block_tables, device),
                context_lens=i32_dev(w.context_lens, device))


def appended_host_cache(orc, w: gen.Workload):
    """The oracle's post-append K/V pools (the state decode attention reads)."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    slots = orc.slot_mapping(w.block_tables, w.context_lens)
    orc.append(w.k_new, w.v_new, slots, kc, vc)
    return kc, vc


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean


def assert_lse_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: -inf pattern differs"
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= LSE_ABS_TOL, f"{what}: lse max abs {err:.3e}"
