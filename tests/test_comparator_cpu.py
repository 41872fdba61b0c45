"""Self-test of the parity gate the GPU tests use (no GPU): outputs the gate
must accept, and corruptions it must reject."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from test_parity_gpu import BF16_MAXABS, BF16_NMSE, F32_MAXABS, compare


def _bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def _ref(seed=0, n=2048):
    rng = np.random.default_rng(seed)
    return rng.normal(0.0, 0.3, size=(16, n // 16))  # 2048 outputs, the Qwen3-1.7B geometry


def test_bf16_rounded_reference_passes():
    ref = _ref()
    maxabs, nmse = compare(_bf16_round(ref), ref, torch.bfloat16)
    assert 0 < maxabs < BF16_MAXABS and 0 < nmse < BF16_NMSE


def test_one_ulp_on_three_elements_moves_the_counts_but_passes():
    ref = _ref(1)
    got = _bf16_round(ref)
    bumped = got.copy()
    idx = [(0, 3), (7, 100), (15, 127)]
    for i, j in idx:
        b = torch.tensor(bumped[i, j]).to(torch.bfloat16)
        bits = b.view(torch.int16) + 1  # next bf16 away from zero (same sign)
        bumped[i, j] = bits.view(torch.bfloat16).double().item()
    assert int((bumped != got).sum()) == 3
    m0, n0 = compare(got, ref, torch.bfloat16)
    m1, n1 = compare(bumped, ref, torch.bfloat16)
    assert n1 > n0 and m1 >= m0


@pytest.mark.parametrize("delta", [0.1, -0.1])
def test_three_elements_off_by_a_tenth_fail_the_bf16_gate(delta):
    ref = _ref(2)
    got = _bf16_round(ref)
    for i, j in [(1, 1), (2, 50), (9, 90)]:
        got[i, j] += delta
    with pytest.raises(AssertionError):
        compare(got, ref, torch.bfloat16)


def test_fp32_gate_is_absolute():
    ref = _ref(3)
    compare(ref + 5e-6, ref, torch.float32)
    with pytest.raises(AssertionError):
        compare(ref + 2 * F32_MAXABS, ref, torch.float32)


def test_non_finite_output_fails():
    ref = _ref(4)
    got = _bf16_round(ref)
    got[3, 3] = np.nan
    with pytest.raises(AssertionError):
        compare(got, ref, torch.bfloat16)
