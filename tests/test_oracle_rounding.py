"""Pins for the oracle's 16-bit rounding of parameters (the storage types of
the mixed-precision step, dl-scratch page 3.4): values worked by hand from the
formats' definitions (bf16: 8 exponent and 7 mantissa bits; IEEE half: 5 and
10), and torch's own conversions on random inputs."""
import numpy as np
import torch

rng = np.random.default_rng(23)


def test_bf16_by_hand(oracle):
    ulp1 = 2.0 ** -7  # spacing of bf16 values in [1, 2)
    x = np.array([1.0, 1 + ulp1 / 2, 1 + 1.5 * ulp1, 1 + ulp1 / 2 + 2.0 ** -20, -3.0, 0.0, 3e38], np.float32)
    want = [1.0, 1.0, 1 + 2 * ulp1, 1 + ulp1, -3.0, 0.0]
    got = oracle.bf16_values(x)
    # ties go to the even mantissa; 3e38 lies between the last two finite values
    assert got[:6].tolist() == want
    assert abs(got[6] - 3e38) <= 2.0 ** 127 * 2.0 ** -8  # within half a bf16 spacing at 2^127


def test_f16_by_hand(oracle):
    ulp1 = 2.0 ** -10  # spacing of half values in [1, 2)
    x = np.array([1.0, 1 + ulp1 / 2, 1 + 1.5 * ulp1, 65504.0, 65519.0, 65520.0, 2.0 ** -24, 2.0 ** -26, -2.0 ** -14],
                 np.float32)
    got = oracle.f16_values(x)
    assert got[:4].tolist() == [1.0, 1.0, 1 + 2 * ulp1, 65504.0]
    assert got[4] == 65504.0 and got[5] == np.inf  # 65520 is the tie above the largest half: to infinity
    assert got[6] == 2.0 ** -24 and got[7] == 0.0 and got[8] == -2.0 ** -14


def test_against_torch_conversions(oracle):
    x = (rng.standard_normal(100_000) * np.exp(rng.uniform(-20, 12, 100_000))).astype(np.float32)
    t = torch.from_numpy(x)
    assert np.array_equal(oracle.bf16_values(x), t.to(torch.bfloat16).double().numpy())
    assert np.array_equal(oracle.f16_values(x), t.to(torch.float16).double().numpy())
