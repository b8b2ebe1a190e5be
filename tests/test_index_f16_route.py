"""The mma.sync index scorer multiplies f16 operands exactly. The bf16 index query of each draft
token is scaled by 2^sigma, which puts its largest |element| in [2^14, 2^15). It is then rounded
to f16. An MXFP4 index-K element becomes the f16 of its E2M1 code times 2^(s_g - max s), the
group's scale relative to the token's largest. A host check covers three things, and so only
the fp32 accumulation rounds:
- every bf16 element within 2^31 of its query's maximum is exact in f16 after the scaling;
- code x 2^rel is exact in f16 for every code and every rel >= -22 (an f16 multiply of two f16s);
- a group more than 2^22 below the largest (dropped) holds less than 2^-19 of that group's
  largest element."""
import numpy as np


def e2m1(code):
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def test_scaled_query_elements_are_exact_in_f16():
    sig8 = 1.0 + np.arange(128) / 128.0                  # every 8-bit bf16 significand
    for E in range(-133, 128):                           # exponent of the query's largest element
        sigma = 14 - E
        for k in range(0, 32):                           # elements 2^0 .. 2^31 below the maximum
            x = np.ldexp(sig8, E - k + sigma)            # the scaled element, exact in fp64
            if E - k < -133:                             # below the smallest bf16
                continue
            assert np.all(x.astype(np.float16).astype(np.float64) == x), (E, k)
        top = np.ldexp(sig8, E + sigma)
        assert np.all((top >= 2.0 ** 14) & (top < 2.0 ** 15))


def test_group_factor_times_code_is_exact_in_f16():
    codes = np.array([e2m1(c) for c in range(16)], np.float16)
    for rel in range(-22, 1):
        f = np.float16(2.0 ** rel)
        assert float(f) == 2.0 ** rel
        prod = codes * f                                 # f16 multiply, one rounding
        assert np.all(prod.astype(np.float64) == codes.astype(np.float64) * 2.0 ** rel), rel


def test_dropped_groups_are_negligible():
    # a group 2^23 or more below the token's largest group scale: |code| <= 6 against a largest
    # group whose largest element is at least 4 x its scale (scale rule 2^(floor(log2 amax) - 2))
    assert 6.0 * 2.0 ** -23 / 4.0 < 2.0 ** -19
