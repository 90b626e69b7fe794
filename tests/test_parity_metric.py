"""The parity metrics themselves: the excess-over-storage-rounding metric is 0
for the correctly rounded oracle, sees a planted error at full size, and equals
the plain metric for fp32 storage."""
import numpy as np
import torch

from tests.helpers import rel_max_err
from tests.parity import bf16_floor, excess_err, storage_round


def test_correctly_rounded_output_has_no_excess():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal(100000) * np.exp(rng.standard_normal(100000))   # heavy tails
    x = storage_round(ref, torch.bfloat16)
    assert excess_err(x, ref, torch.bfloat16) <= 1e-15
    assert rel_max_err(x, ref) == bf16_floor(ref) > 2e-2    # the plain metric would fail


def test_planted_error_is_seen_in_full():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal(10000)
    rms = np.sqrt(np.mean(ref ** 2))
    x = storage_round(ref, torch.bfloat16)
    i = int(np.argmin(np.abs(ref)))            # an element whose own rounding is tiny
    x[i] += 0.05 * rms
    assert abs(excess_err(x, ref, torch.bfloat16) - 0.05) < 2e-3


def test_fp32_storage_is_the_plain_metric():
    rng = np.random.default_rng(2)
    ref = rng.standard_normal(1000)
    x = ref + 1e-5 * rng.standard_normal(1000)
    assert abs(excess_err(x, ref, torch.float32) - rel_max_err(x, ref)) < 1e-6
