"""CPU checks of the parity helpers: the output-rounding allowance bounds the rounding of
fp32 values to bf16 / fp16 (one rounding, as the kernels do) and is zero for other types."""
import numpy as np
import torch

from tests.parity_util import compare, half_ulp


def test_half_ulp_bounds_one_rounding():
    x32 = torch.tensor(np.random.default_rng(0).normal(size=200000) * 5, dtype=torch.float32)
    x = x32.double().numpy()
    for dt in (torch.bfloat16, torch.float16):
        r = x32.to(dt).double().numpy()
        assert np.all(np.abs(r - x) <= half_ulp(x, dt))
    assert np.all(half_ulp(x, torch.float32) == 0.0)
    assert half_ulp(np.array([3.0]), torch.bfloat16)[0] == 2.0 ** -7


def test_compare_charges_only_error_beyond_rounding():
    o_ref = np.array([[3.0 + 0.0078]])          # an exact result just under half a bf16 ulp
    o = torch.tensor([[3.0]], dtype=torch.bfloat16)
    lse = torch.zeros(1)
    compare(o, lse, o_ref, np.zeros(1), "within rounding")
    try:
        compare(torch.tensor([[3.03125]], dtype=torch.bfloat16), lse, o_ref, np.zeros(1), "off")
    except AssertionError:
        pass
    else:
        raise AssertionError("an error of two bf16 ulps at 3 must fail")
