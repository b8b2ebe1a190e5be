"""The tensor-core attention widens MXFP4 V to bf16 without a float round trip. It takes the f16
of each E2M1 code, shifts that f16's exponent and mantissa bits down by 3, and reads the result
as a bf16 holding the code x 2^-112. Two bf16 multiplies by powers of two, whose product is
2^(b - 15), then apply the E8M0 byte b. A host model of that bit route must give exactly code x
2^(b - 127) rounded to bf16, for all 16 codes and every scale byte b < 255. Each factor must be a
normal bf16, and b = 255 (E8M0 NaN) must give NaN. The E2M1 values come from the OCP MX
definition, and the bf16 multiplies are torch's (one rounding each)."""
import numpy as np
import torch


def e2m1(code):
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def bf16_from_bits(bits):
    return torch.tensor(np.array(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def factors(b):
    k = b - 15
    k1 = k >> 1
    k2 = k - k1
    return k1, k2


def test_bit_route_is_exact_for_every_code_and_scale():
    codes = np.arange(16)
    f16 = np.array([e2m1(c) for c in codes], np.float16).view(np.uint16).astype(np.uint32)
    shifted = ((f16 & 0x7FFF) >> 3) | (f16 & 0x8000)
    x = bf16_from_bits(shifted)
    assert torch.equal(x.to(torch.float64), torch.tensor([e2m1(c) * 2.0 ** -112 for c in codes], dtype=torch.float64))
    for b in range(255):
        k1, k2 = factors(b)
        assert -126 <= k1 <= 127 and -126 <= k2 <= 127          # normal bf16 powers of two
        assert k1 + k2 == b - 15
        s1 = torch.tensor([2.0 ** k1], dtype=torch.bfloat16)
        s2 = torch.tensor([2.0 ** k2], dtype=torch.bfloat16)
        got = ((x * s1) * s2).to(torch.float64)
        want = torch.tensor([e2m1(c) * 2.0 ** (b - 127) for c in codes], dtype=torch.float64)
        want = want.to(torch.bfloat16).to(torch.float64)
        assert torch.equal(got, want), b


def test_nan_scale_gives_nan():
    s1 = bf16_from_bits([0x7FC0])                               # the factor used for b = 255
    x = bf16_from_bits([0x0000, 0x3F80 >> 3])
    assert torch.all(torch.isnan(x * s1))
