"""Pins of the oracle's element formats and quantisers against things other than itself:
closed forms from the OCP specs, torch's float8_e4m3fn / bfloat16 conversions, brute force
over all codes, and hand-derived golden rows (tests/golden/)."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hexf(s):
    s = s.strip()
    if s in ("inf", "-inf", "nan", "-nan"):
        v = float(s.lstrip("-"))
        return -v if s.startswith("-") else v
    return float.fromhex(s)


# ---- tables ------------------------------------------------------------------------------
def test_e2m1_table_closed_form():
    # OCP MX v1.0 E2M1: exponent bias 1; exponent field 0 is subnormal (0.5 * m).
    for nib in range(16):
        s, e, m = nib >> 3, (nib >> 1) & 3, nib & 1
        v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        v = -v if s else v
        got = oracle.e2m1_value(nib)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), nib


def test_e8m0_closed_form():
    for b in range(255):
        assert oracle.e8m0_value(b) == 2.0 ** (b - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_bf16_value_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# ---- E2M1 encoder: brute force ------------------------------------------------------------
MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def brute_e2m1(v):
    a = Fraction(abs(v))                     # exact distances
    best = None
    for c in range(8):                       # nearest magnitude; on a tie the even code
        d = abs(a - Fraction(MAGS[c]))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return (8 if math.copysign(1, v) < 0 else 0) | best[1]


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(0)
    vals = list(rng.uniform(-8, 8, 5000)) + [m + d for m in
                                             [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0]
                                             for d in (-1e-9, 0.0, 1e-9)]
    vals += [-x for x in vals] + [0.0, -0.0, 100.0, -1e30]
    for v in vals:
        assert oracle.e2m1_encode(v) == brute_e2m1(v), v


# ---- MXFP4 row quantiser --------------------------------------------------------------------
def floor_log2(a):
    e = 0
    while 2.0 ** e > a:
        e -= 1
    while 2.0 ** (e + 1) <= a:
        e += 1
    return e


def brute_mxfp4_row(x):
    """Per group: the scale from the benchmark rule computed by search, then every element's
    code by brute force over all codes."""
    x = np.asarray(x, np.float32).astype(np.float64)
    codes, scales = [], []
    for g in range(4):
        xg = x[32 * g:32 * g + 32]
        amax = float(np.max(np.abs(xg)))
        se = 0 if amax == 0 else min(127, max(-127, floor_log2(amax) - 2))
        scales.append(se + 127)
        codes += [brute_e2m1(float(v) / 2.0 ** se) for v in xg]
    nib = np.array([codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(64)], np.uint8)
    return nib, np.array(scales, np.uint8)


def test_mxfp4_quant_brute_force():
    rng = np.random.default_rng(1)
    rows = [rng.standard_normal(128).astype(np.float32) * s for s in (1, 50, 1e-3, 3e5, 1e-38)]
    rows.append(np.zeros(128, np.float32))
    rows.append(np.where(rng.random(128) < 0.5, 0, rng.standard_normal(128)).astype(np.float32))
    for x in rows:
        nib, sc = oracle.mxfp4_quant_row(x)
        bn, bs = brute_mxfp4_row(x)
        assert np.array_equal(sc, bs)
        assert np.array_equal(nib, bn)


def test_mxfp4_golden_row():
    x = np.zeros(128, np.float32)
    exp_codes = np.zeros(128, np.int64)
    exp_scales = {}
    for line in open(os.path.join(GOLDEN, "mxfp4_row.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        if line[0] == "scale":
            exp_scales[int(line[1])] = int(line[2])
            continue
        i, v, c = int(line[0]), _hexf(line[1]), int(line[2], 16)
        assert np.float32(v) == v, "golden value must be exact in fp32"
        x[i] = v
        exp_codes[i] = c
    nib, sc = oracle.mxfp4_quant_row(x)
    assert [int(s) for s in sc] == [exp_scales[g] for g in range(4)]
    got_codes = np.stack([nib & 0xF, nib >> 4], axis=1).reshape(-1)
    assert np.array_equal(got_codes, exp_codes)


def test_mxfp4_dequant_of_golden_row_and_nibble_order():
    # A page holding one row whose element 2i has code 0x2 (+1.0) in the low nibble and
    # element 2i+1 code 0xC (-2.0) in the high nibble, scale bytes 126, 127, 128, 129.
    page = np.zeros(8704, np.uint8)
    page[5 * 64:6 * 64] = 0xC2
    page[8192 + 5 * 4:8192 + 6 * 4] = [126, 127, 128, 129]
    row = oracle.mxfp4_load_row(page, 5)
    for d in range(128):
        s = 2.0 ** (d // 32 - 1)
        assert row[d] == (1.0 * s if d % 2 == 0 else -2.0 * s)


def test_mxfp4_idempotent():
    rng = np.random.default_rng(2)
    for scale in (1.0, 50.0, 1e-4):
        x = (rng.standard_normal(128) * scale).astype(np.float32)
        nib, sc = oracle.mxfp4_quant_row(x)
        page = np.zeros(8704, np.uint8)
        page[:64] = nib
        page[8192:8196] = sc
        y = oracle.mxfp4_load_row(page, 0).astype(np.float32)
        nib2, sc2 = oracle.mxfp4_quant_row(y)
        # requantising gives the same codes; the scale byte may only drop when the group's
        # amax rounded down below a power of two, so compare dequantised values instead
        page2 = np.zeros(8704, np.uint8)
        page2[:64] = nib2
        page2[8192:8196] = sc2
        assert np.array_equal(oracle.mxfp4_load_row(page2, 0), y.astype(np.float64))


def test_mxfp4_nonfinite_group():
    x = np.ones(128, np.float32)
    x[40] = np.nan
    x[100] = np.inf
    nib, sc = oracle.mxfp4_quant_row(x)
    assert list(sc) == [125, 0xFF, 125, 0xFF]
    assert np.all(nib[16:32] == 0) and np.all(nib[48:64] == 0)


# ---- e4m3: pack_q and the row-scale quantiser ----------------------------------------------
def test_pack_q_golden():
    for line in open(os.path.join(GOLDEN, "e4m3_pack.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        v, b = _hexf(line[0]), int(line[1], 16)
        assert int(oracle.pack_q_e4m3(np.array([v], np.float32))[0]) == b, line


def test_pack_q_in_range_equals_torch_cast():
    # every e4m3 value, every midpoint between neighbours, and +-1 fp32 ulp around each
    vals = np.array([oracle.e4m3_value(b) for b in range(256)])
    vals = np.sort(vals[np.isfinite(vals)])
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)),
                          np.nextafter(pts, np.float32(-np.inf))])
    rng = np.random.default_rng(3)
    pts = np.concatenate([pts, rng.standard_normal(20000).astype(np.float32) * 30,
                          (rng.standard_normal(5000) * 1e-3).astype(np.float32)])
    pts = pts[np.abs(pts) <= 448]
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.pack_q_e4m3(pts)
    assert np.array_equal(got, ref)


def test_pack_q_saturates_and_nan():
    x = np.array([448.0, 448.5, 464.0, 465.0, 1e38, np.inf, -np.inf, -449.0, np.nan, -np.nan],
                 np.float32)
    got = oracle.pack_q_e4m3(x)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x7F]


def test_e4m3_rowscale_row():
    rng = np.random.default_rng(4)
    for scale in (1.0, 50.0, 1e-3):
        x = (rng.standard_normal(128) * scale).astype(np.float32)
        codes, s = oracle.e4m3rs_quant_row(x)
        s_ref = np.float32(np.max(np.abs(x))) / np.float32(448.0)     # fp32 division
        assert np.float32(s) == s_ref
        y = (x / s_ref).astype(np.float32)
        ref = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
        assert np.array_equal(codes, ref.numpy())
        page = np.zeros(16896, np.uint8)
        page[:128] = codes
        page[16384:16388] = np.frombuffer(np.float32(s).tobytes(), np.uint8)
        back = oracle.e4m3rs_load_row(page, 0)
        assert np.array_equal(back, torch.from_numpy(codes).view(torch.float8_e4m3fn)
                              .to(torch.float64).numpy() * float(s))
    codes, s = oracle.e4m3rs_quant_row(np.zeros(128, np.float32))
    assert s == 1.0 and np.all(codes == 0)


def _e4m3_cast(y):
    return torch.from_numpy(np.clip(y, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rowscale_divides_by_the_scale():
    """Codes are the e4m3 cast of fl32(x / s), a true fp32 division: elements placed within a few
    ulps of e4m3 rounding midpoints, where x * fl32(1 / s) would land on another code."""
    rng = np.random.default_rng(41)
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (grid[1:] + grid[:-1]) / 2                               # e4m3 rounding boundaries
    n_disc = 0
    for _ in range(24):
        amax = np.float32(rng.uniform(0.5, 8.0) * 2.0 ** rng.integers(-8, 8))
        s = np.float32(amax) / np.float32(448.0)
        x = np.empty(128, np.float32)
        x[0] = amax
        m = rng.choice(mids[mids > 1.0], size=127)
        base = (m * np.float64(s)).astype(np.float32)
        steps = rng.integers(-2, 3, size=127)
        for i in range(127):
            v = base[i]
            for _ in range(abs(int(steps[i]))):
                v = np.nextafter(v, np.float32(np.inf if steps[i] > 0 else -np.inf), dtype=np.float32)
            x[i + 1] = -v if rng.random() < 0.5 else v
        x = np.clip(x, -amax, amax)
        codes, s_o = oracle.e4m3rs_quant_row(x)
        assert np.float32(s_o) == s
        want = _e4m3_cast((x / s).astype(np.float32))
        assert np.array_equal(codes, want)
        n_disc += int(np.sum(_e4m3_cast((x * (np.float32(1.0) / s)).astype(np.float32)) != want))
    assert n_disc > 0, "no element separates division from the reciprocal product"
