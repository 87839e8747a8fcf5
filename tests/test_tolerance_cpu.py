"""The parity bar the GPU tests apply (tests/gpu_common.compare), checked on
hand-made arrays: 1e-2 absolute below |ref| = 2, 1e-2 beyond half a bf16 ulp
of ref from 2 up, 2e-2 per-row normwise, 2e-3 on lse."""
import numpy as np
import pytest
import torch

from tests.gpu_common import compare


def _row(values):
    return np.asarray([values], dtype=np.float64)


def test_small_outputs_get_the_bar_as_it_stands():
    ref = _row([1.5, 0.25, -0.5])
    compare(torch.tensor(ref + 0.0099), ref)
    with pytest.raises(AssertionError):
        compare(torch.tensor(ref + [[0.011, 0, 0]]), ref)


def test_outputs_from_two_up_are_not_charged_their_bf16_rounding():
    ref = _row([3.0, 0.25, -5.0])          # half ulp: 2^-7 at 3, 2^-6 at 5
    compare(torch.tensor(ref + [[0.0175, 0, 0]]), ref)
    compare(torch.tensor(ref + [[0, 0, -0.0255]]), ref)
    with pytest.raises(AssertionError):
        compare(torch.tensor(ref + [[0.0185, 0, 0]]), ref)
    with pytest.raises(AssertionError):
        compare(torch.tensor(ref + [[0, 0.0101, 0]]), ref)


def test_row_relative_and_lse_bars():
    ref = _row([0.2, 0.1, 0.05])
    with pytest.raises(AssertionError):              # 0.005 / 0.2 = 2.5e-2 > 2e-2
        compare(torch.tensor(ref + [[0.005, 0, 0]]), ref)
    lse = np.array([1.0])
    compare(torch.tensor(ref), ref, torch.tensor(lse + 0.0019), lse)
    with pytest.raises(AssertionError):
        compare(torch.tensor(ref), ref, torch.tensor(lse + 0.0021), lse)
