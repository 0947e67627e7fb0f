"""CPU checks of the parity helpers: the output-rounding allowance bounds the rounding of
fp32 values to bf16 / fp16 (one rounding, as the kernels do) and is zero for other types;
without the allowance the bounds apply to the raw differences."""
import numpy as np
import pytest
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


def test_compare_charges_only_error_beyond_rounding_with_the_allowance():
    o_ref = np.array([[3.0 + 0.0078]])          # an exact result just under half a bf16 ulp
    o = torch.tensor([[3.0]], dtype=torch.bfloat16)
    lse = torch.zeros(1)
    compare(o, lse, o_ref, np.zeros(1), "within rounding", allowance=True)
    with pytest.raises(AssertionError):
        compare(torch.tensor([[3.03125]], dtype=torch.bfloat16), lse, o_ref, np.zeros(1),
                "off", allowance=True)


def test_compare_is_raw_by_default():
    o_ref = np.array([[3.0 + 0.0078], [0.0]])   # the same row: raw error 0.0078 <= 1e-2 ...
    o = torch.tensor([[3.0], [0.0]], dtype=torch.bfloat16)
    lse = torch.zeros(2)
    with pytest.raises(AssertionError, match="mean"):  # ... but a mean of 3.9e-3 > 1e-3
        compare(o, lse, o_ref, np.zeros(2), "raw")
    stats = compare(o, lse, o_ref, np.zeros(2), "adjusted", allowance=True)
    assert stats["raw_max_abs_o"] == pytest.approx(0.0078)
    assert stats["max_abs_o"] == 0.0


def test_compare_logs_raw_and_adjusted(tmp_path, monkeypatch):
    import json
    log = tmp_path / "parity.jsonl"
    monkeypatch.setenv("FA_PARITY_LOG", str(log))
    o = torch.tensor([[0.5, -0.25]], dtype=torch.bfloat16)
    compare(o, torch.zeros(1), np.array([[0.5, -0.2505]]), np.array([1e-4]), "logged")
    rec = json.loads(log.read_text().splitlines()[-1])
    assert rec["what"] == "logged" and rec["allowance"] is False
    assert rec["raw_max_abs_o"] == pytest.approx(5e-4)
    assert rec["max_abs_lse"] == pytest.approx(1e-4)
