"""CPU check of the FMA-pipe exp2 used for part of the softmax: the same
float32 operation sequence as exp2_poly_x2 in csrc/ptx.cuh, emulated with
numpy float32, must stay within the polynomial's stated bound of 2^x (well
under bf16's half-ulp) over the whole input range the kernel feeds it, and
give exactly 0-ish below the clamp."""
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "attention_all_layout_gb300", "csrc")


def coefficients():
    txt = open(os.path.join(CSRC, "exp2_poly.cuh")).read()
    c = [np.float32(float(x)) for x in re.findall(r"kExp2C\d = ([-0-9.e+]+)f;", txt)]
    bound = float(re.search(r"kExp2PolyMaxRelErr = ([-0-9.e+]+)f;", txt).group(1))
    return c, bound


def exp2_poly_emulated(x):
    c0, c1, c2, c3 = coefficients()[0]
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-126.0))
    t = (x + f32(12582912.0)).astype(f32)
    j = (t - f32(12582912.0)).astype(f32)
    f = (x - j).astype(f32)  # the kernel's fma(j, -1, x) is exact here as well
    p = (f * c3 + c2).astype(f32)
    p = (p * f + c1).astype(f32)
    p = (p * f + c0).astype(f32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.view(np.float32)


def test_relative_error_within_bound():
    _, bound = coefficients()
    x = np.concatenate([np.linspace(-120, 8, 2_000_001), np.arange(-120, 9).astype(np.float64) + 0.5])
    x = x.astype(np.float32)
    y = exp2_poly_emulated(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1)
    assert rel.max() <= bound * 1.05 + 2e-7
    assert rel.max() < 2 ** -9  # far inside bf16's rounding


def test_clamp_gives_negligible_values():
    y = exp2_poly_emulated(np.array([-126.0, -200.0, -1e30, -np.inf], dtype=np.float32))
    assert np.all(y >= 0) and np.all(y < 2.0 ** -124)


def test_zero_and_integers_are_close():
    x = np.arange(-20, 9, dtype=np.float32)
    y = exp2_poly_emulated(x).astype(np.float64)
    np.testing.assert_allclose(y, np.exp2(x.astype(np.float64)), rtol=1e-4)
