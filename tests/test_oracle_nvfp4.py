"""Pins of the oracle's NVFP4 pages against things other than itself: hand-derived golden rows
(tests/golden/nvfp4_row.txt), exact round trips of values the format represents, brute force over
all sixteen E2M1 codes with torch's float8_e4m3fn cast choosing the block scale, the decode as a
product of the OCP tables, and closed-form page scores and attention over NVFP4 pools.

NVFP4 as the pages name it ("Mono decode over the MXFP4 KV and index caches", PR title "FP4
index cache and NVFP4 sparse KV cache"; commit "--index-cache-dtype mxfp4": "NVFP4 main KV,
NVFP4 index ... stay refused"): E2M1 elements, one E4M3 scale per 16 elements, one fp32
per-tensor decode scale g. The page layout and rounding are readings (orc_nvfp4_quant_row)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import helpers as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])   # OCP MX v1.0 magnitudes


def _codes(nib):
    nib = np.asarray(nib, np.uint8)
    out = np.empty(128, np.uint8)
    out[0::2] = nib & 0xF
    out[1::2] = nib >> 4
    return out


def _hexf(s):
    if s in ("inf", "-inf", "nan"):
        return float(s)
    return float.fromhex(s)


def _golden_rows():
    rows, cur = [], None
    for line in open(os.path.join(GOLDEN, "nvfp4_row.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "row":
            cur = dict(name=f[1], g=float.fromhex(f[3]), x=np.zeros(128, np.float32),
                       scale=np.zeros(8, np.uint8), code=np.zeros(128, np.uint8))
            rows.append(cur)
        elif f[0] == "scale":
            cur["scale"][int(f[1])] = int(f[2], 16)
        else:
            i, v, c = int(f[0]), _hexf(f[1]), int(f[2], 16)
            assert math.isnan(v) or np.float32(v) == v, "golden value must be exact in fp32"
            cur["x"][i] = v
            cur["code"][i] = c
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r["name"])
def test_nvfp4_golden_rows(row):
    nib, sc = oracle.nvfp4_quant_row(row["x"], row["g"])
    assert [hex(b) for b in sc] == [hex(b) for b in row["scale"]]
    got = _codes(nib)
    bad = np.nonzero(got != row["code"])[0]
    assert bad.size == 0, [(int(i), hex(got[i]), hex(row["code"][i])) for i in bad]


def test_nvfp4_round_trip_of_representable_values():
    # Blocks whose largest element is E2M1 6 times E4M3(b) times g (g a power of two): then
    # amax / (6 g) is E4M3(b) exactly, the block's byte is b and every x / S is the E2M1 value
    # itself, so the codes come back unchanged.
    rng = np.random.default_rng(11)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    normal_bytes = [b for b in range(0x08, 0x7F)]   # normal, finite, positive
    for trial in range(200):
        g = 2.0 ** int(rng.integers(-12, 4))
        codes = rng.integers(0, 16, 128).astype(np.uint8)
        bytes_ = rng.choice(normal_bytes, 8).astype(np.uint8)
        for blk in range(8):
            codes[16 * blk + int(rng.integers(0, 16))] = 0x7 | (int(rng.integers(0, 2)) << 3)   # +-6
        x = np.empty(128, np.float32)
        for i in range(128):
            v = E2M1[codes[i] & 7] * e4m3[bytes_[i // 16]] * g
            x[i] = -v if codes[i] & 8 else v
            assert np.float32(x[i]) == (-v if codes[i] & 8 else v)
        nib, sc = oracle.nvfp4_quant_row(x, g)
        assert np.array_equal(sc, bytes_), trial
        assert np.array_equal(_codes(nib), codes), trial


def _brute_force_row(x, g):
    """Scale bytes by torch's float8_e4m3fn cast (round to nearest even) of the fp32 quotient
    clamped to 448; codes by the nearest of all sixteen E2M1 values to the fp32 x / S, ties to
    the even code, |y| above 6 saturating, the sign of x kept."""
    x = np.asarray(x, np.float32)
    six_g = np.float32(6.0) * np.float32(g)
    scale = np.zeros(8, np.uint8)
    codes = np.zeros(128, np.uint8)
    for blk in range(8):
        xb = x[16 * blk:16 * blk + 16]
        if not np.all(np.isfinite(xb)):
            scale[blk] = 0x7F
            continue
        s = np.float32(np.max(np.abs(xb))) / six_g
        s = min(float(s), 448.0)
        b = int(torch.tensor([s], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
        scale[blk] = b
        S = np.float32(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)[0]) * np.float32(g)
        if S == 0:
            continue
        for i in range(16):
            y = float(np.float32(xb[i]) / S)
            a = abs(y)
            d = np.abs(E2M1 - a)
            best = np.nonzero(d == d.min())[0]
            c = int(best[0]) if len(best) == 1 else int(best[0] if best[0] % 2 == 0 else best[1])
            if a > 6.0:
                c = 7
            codes[16 * blk + i] = c | (8 if math.copysign(1.0, y) < 0 else 0)
    return scale, codes


@pytest.mark.parametrize("seed", range(6))
def test_nvfp4_codes_are_the_nearest_by_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    for trial in range(40):
        g = float(np.float32(10.0 ** rng.uniform(-3, 1)))
        spread = 10.0 ** rng.uniform(-3, 3, 8).repeat(16)
        x = (rng.standard_normal(128) * spread).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(0, 128)] = np.float32(0.0) * -1.0
        nib, sc = oracle.nvfp4_quant_row(x, g)
        ref_sc, ref_codes = _brute_force_row(x, g)
        assert np.array_equal(sc, ref_sc), (seed, trial)
        assert np.array_equal(_codes(nib), ref_codes), (seed, trial)


def test_nvfp4_page_row_decode_is_the_product_of_the_tables():
    rng = np.random.default_rng(5)
    page = rng.integers(0, 256, wl.NVFP4_PAGE_BYTES, dtype=np.uint8)
    e4m3 = torch.from_numpy(page[8192:].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    g = float(np.float32(0.0173))
    for slot in (0, 1, 77, 127):
        got = oracle.nvfp4_load_row(page, slot, g)
        codes = _codes(page[slot * 64:slot * 64 + 64])
        for d in range(128):
            c = codes[d]
            v = E2M1[c & 7] * (-1 if c & 8 else 1) * e4m3[slot * 8 + d // 16] * g
            if math.isnan(v):
                assert math.isnan(got[d])
            else:
                assert got[d] == v, (slot, d)


def test_nvfp4_page_scales_follow_the_nibble_rows():
    # the row store: nibbles of slot s at 64 s, its eight block scales at 8192 + 8 s
    w = wl.Workload("nv_layout", B=1, Q=1, Hq=8, Hkv=1, max_ctx=256, topk=2, num_splits=1, seed=3,
                    kv_format=wl.KV_NVFP4, idx_format=wl.KV_NVFP4, nv_scale_k=0.25, nv_scale_v=0.5,
                    nv_scale_idx=0.125)
    sh = oracle.shape_of(w)
    k_pool, v_pool, idx_pool = wl.empty_pools(w)
    assert idx_pool.shape[1] == wl.NVFP4_PAGE_BYTES and k_pool.shape[2] == wl.NVFP4_PAGE_BYTES
    rng = np.random.default_rng(9)
    T = 200
    k = rng.standard_normal((1, T, 1, 128)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, 128)).astype(np.float32)
    kidx = rng.standard_normal((1, T, 128)).astype(np.float32)
    pt = np.array([[1, 0]], np.int32)
    oracle.kv_fill(sh, k, v, kidx, pt, np.array([T], np.int32), k_pool, v_pool, idx_pool)
    for pos in (0, 5, 127, 128, 199):
        phys, slot = pt[0, pos // 128], pos % 128
        for pool, x, g in ((k_pool[:, 0], k[0, pos, 0], 0.25), (v_pool[:, 0], v[0, pos, 0], 0.5),
                           (idx_pool, kidx[0, pos], 0.125)):
            nib, sc = oracle.nvfp4_quant_row(x, g)
            page = pool[phys]
            assert np.array_equal(page[slot * 64:slot * 64 + 64], nib)
            assert np.array_equal(page[8192 + slot * 8:8192 + slot * 8 + 8], sc)


def test_nvfp4_index_score_closed_form():
    # One page, every token row the same known NVFP4 row; a one-hot query on dimension d scores
    # each token E2M1 x E4M3 x g_idx of that dimension: the page score is that product.
    g = 0.0625
    w = wl.Workload("nv_score", B=1, Q=1, Hq=8, Hkv=1, max_ctx=128, topk=1, num_splits=1, seed=1,
                    kv_format=wl.KV_NVFP4, idx_format=wl.KV_NVFP4, nv_scale_idx=g, nv_scale_k=4.0)
    sh = oracle.shape_of(w)
    _, _, idx_pool = wl.empty_pools(w)
    x = np.linspace(-3.0, 5.0, 128).astype(np.float32)
    nib, sc = oracle.nvfp4_quant_row(x, g)
    for slot in range(128):
        idx_pool[0, slot * 64:slot * 64 + 64] = nib
        idx_pool[0, 8192 + slot * 8:8192 + slot * 8 + 8] = sc
    e4m3 = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = _codes(nib)
    for d in (0, 17, 64, 127):
        q = np.zeros((1, 1, 128), np.float32)
        q[0, 0, d] = 1.0
        qb = wl.f32_to_bf16_bits(q)
        s = oracle.index_scores(sh, qb, idx_pool, np.array([[0]], np.int32), np.array([128], np.int32))
        c = codes[d]
        want = E2M1[c & 7] * (-1 if c & 8 else 1) * e4m3[d // 16] * g
        assert s[0, 0] == want, (d, s[0, 0], want)


@pytest.mark.parametrize("kv_scale", [(0.0173, 0.0173), (0.03125, 0.5)])
def test_nvfp4_attention_matches_dense_softmax(kv_scale):
    # the oracle's whole step over NVFP4 pools against torch float64 softmax attention over the
    # decoded selected tokens (the selection the oracle made)
    w = wl.Workload("nv_attn", B=2, Q=4, Hq=8, Hkv=2, max_ctx=700, topk=3, num_splits=2, seed=21, ragged=True,
                    kv_format=wl.KV_NVFP4, idx_format=wl.KV_NVFP4, nv_scale_k=kv_scale[0], nv_scale_v=kv_scale[1])
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    res, new_pools = H.oracle_step(w, data, pools)
    q = H.q_values(w, data, res)
    ref = H.dense_selected_attention(w, data, q, new_pools[0], new_pools[1], res["topk_pages"], res["topk_count"])
    assert np.allclose(res["out"], ref, rtol=1e-12, atol=1e-12)
