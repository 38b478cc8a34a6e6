"""The parity metric itself: rounding the exact value to bf16 costs nothing,
while an error of one bf16 ulp on top of the rounding is counted."""
import numpy as np
import torch

from _common import half_ulp_bf16, rel_max


def test_correct_rounding_is_free_and_real_errors_count():
    rng = np.random.RandomState(0)
    ref = rng.standard_t(3, size=100000) * 3.0  # heavy tails, like the gate gradients
    rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert rel_max(rounded, ref, bf16=True) == 0.0
    assert rel_max(rounded, ref, bf16=False) > 1e-2  # why plain max-norm cannot apply to bf16 storage
    i = np.argmax(np.abs(ref))
    bad = rounded.copy()
    bad[i] += 4 * half_ulp_bf16(ref[i])  # two ulps off at the largest element
    assert rel_max(bad, ref, bf16=True) > 1e-2
