"""The tensor-core index scorer feeds the bf16 index query to a block-scaled e4m3 MMA as two e4m3
pieces, p0 = e4m3(x) and p1 = e4m3(x - p0), both rounded to nearest even, after the group's largest
|x| is scaled into (224, 448]. A host check over every bf16 value of magnitude up to 448 shows
three things. The pieces stay finite. The split is exact for |x| >= 1/4, which is within 2^9.8 of
a group maximum above 224. A smaller element is off by at most half the e4m3 subnormal step,
2^-10, which is 2^-17.8 of the group maximum. The e4m3 rounding is torch's float8_e4m3fn cast."""
import math

import numpy as np
import torch


def e4m3(x64):
    return torch.from_numpy(x64.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_two_piece_split_of_every_bf16_up_to_448():
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = torch.from_numpy((bits.astype(np.uint16)).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    p0 = e4m3(x)
    p1 = e4m3(x - p0)                      # x - p0 is exact in fp64
    assert np.all(np.isfinite(p0)) and np.all(np.isfinite(p1))
    err = np.abs(x - p0 - p1)
    assert np.all(err[np.abs(x) >= 0.25] == 0.0)
    assert err.max() <= 2.0 ** -10
    # relative to the group maximum (> 224 after scaling), and the 1/4 threshold relative to it
    assert 2.0 ** -10 / 224.0 <= 2.0 ** -17.8
    assert math.log2(448.0 / 0.25) <= 10.81 and math.log2(224.0 / 0.25) >= 9.8
