"""The polynomial exp2 of the prefill softmax (Cody-Waite range reduction and a
degree-3 Remez fit), evaluated step by step in float32 as the kernel does,
against the exact 2^t: relative error within the fit's bound plus float32
rounding, on the softmax's input range t in [-125, 8]. CPU only."""
import os
import re
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "paged_kv_decode_gb300", "csrc")


def kernel_coefficients():
    src = open(os.path.join(CSRC, "prefill.cu")).read()
    m = re.search(r"c0 = ([0-9.e+-]+)f, c1 = ([0-9.e+-]+)f, c2 = ([0-9.e+-]+)f,\s*c3 = ([0-9.e+-]+)f", src)
    return [np.float32(float(x)) for x in m.groups()]


def exp2_poly_f32(t):
    c0, c1, c2, c3 = kernel_coefficients()
    f32 = np.float32
    t = np.maximum(t.astype(np.float32), f32(-125.0))
    j = (t + f32(12582912.0)).astype(np.float32)
    n = (j - f32(12582912.0)).astype(np.float32)
    f = (t - n).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = p.view(np.int32) + (j.view(np.int32) << 23)
    return bits.view(np.float32)


def test_kernel_constants_match_the_fit():
    sys.path.insert(0, CSRC)
    from exp2_poly_fit import remez_exp2

    coeffs, max_rel = remez_exp2()
    assert max_rel < 8e-5
    np.testing.assert_allclose(kernel_coefficients(), coeffs.astype(np.float32), rtol=0, atol=1e-7)


def test_relative_error_over_the_softmax_range():
    t = np.concatenate([np.linspace(-125, 8, 2_000_001), np.arange(-125, 9, dtype=np.float64)])
    got = exp2_poly_f32(t).astype(np.float64)
    want = np.exp2(t.astype(np.float32).astype(np.float64))
    rel = np.abs(got / want - 1)
    assert rel.max() < 7.5e-5 + 4 * 2.0 ** -24
    # -inf (masked scores) gives a negligible positive weight, not NaN
    assert 0 <= exp2_poly_f32(np.array([-np.inf]))[0] < 1e-37
