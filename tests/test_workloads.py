"""The seeded input recipe against the benchmark workloads' definitions (host only): the four fixed
workloads and the 216-case sweep, generated shapes and structure (ragged lengths, the page table,
the new rows, rows scaled x50, shifted index-K pages, poisoned tail slots), bf16 rounding against
torch, and determinism."""
import itertools

import numpy as np
import torch

from sparse_attention_decode_mxfp4_gb300 import workloads as wl


def test_fixed_workloads_match_their_definitions():
    c1, c2, c3, c4 = (wl.config(n) for n in (1, 2, 3, 4))
    assert (c1.B, c1.Q, c1.Hq, c1.Hkv, c1.max_ctx, c1.topk, c1.num_splits) == (1, 1, 8, 1, 1024, 4, 2)
    assert (c2.B, c2.Q, c2.Hq, c2.Hkv, c2.max_ctx, c2.topk, c2.num_splits) == (4, 8, 16, 1, 16384, 16, 4)
    assert c2.kv_format == wl.KV_MXFP4 and c2.max_pages == 128
    assert (c3.B, c3.Q, c3.Hq, c3.max_ctx, c3.topk, c3.num_splits) == (4, 8, 16, 65536, 32, 8)
    assert c3.kv_format == wl.KV_E4M3_ROWSCALE and c3.big_row_frac == 0.01 and c3.big_row_factor == 50.0
    assert (c4.B, c4.Q, c4.Hq, c4.topk, c4.num_splits) == (2, 8, 16, 64, 16)
    assert c4.ctx_lens == (245707, 245707) and c4.max_pages == 1920
    assert 245707 == 1919 * 128 + 75 and 1920 * 128 - 245707 == 53     # 53 tail slots
    assert c4.shift_page_frac == 0.05 and c4.shift_value == 3.0
    assert [c.seed for c in (c1, c2, c3, c4)] == [1001, 1002, 1003, 1004]


def test_sweep_is_the_full_product():
    cases = wl.sweep_cases()
    assert len(cases) == 216
    assert [c.seed for c in cases] == list(range(5000, 5216))
    axes = {(c.B, c.Q, c.max_ctx, c.topk, c.Hq) for c in cases}
    assert axes == set(itertools.product(wl.SWEEP_B, wl.SWEEP_Q, wl.SWEEP_CTX, wl.SWEEP_K, wl.SWEEP_HQ))
    assert all(c.ragged and c.Hkv == 1 for c in cases)
    # every (B, Q, ctx) has a case with more partitions than selected pages
    for key in itertools.product(wl.SWEEP_B, wl.SWEEP_Q, wl.SWEEP_CTX):
        assert any(c.num_splits > c.topk for c in cases if (c.B, c.Q, c.max_ctx) == key)


def test_generated_shapes_rows_and_page_table():
    w = wl.shrink(wl.config(2), B=3, max_ctx=3000, ragged=True, seed=77)
    d = wl.generate(w)
    ctx = d["ctx_len"]
    assert ctx.dtype == np.int32 and np.all(ctx >= w.Q) and np.all(ctx <= w.max_ctx)
    assert np.all(ctx >= np.floor(0.5 * w.max_ctx))
    T = int(ctx.max())
    assert d["k"].shape == (3, T, 1, 128) and d["kidx"].shape == (3, T, 128)
    assert d["q"].shape == (3, 8, 16, 128) and d["qidx_bf16"].shape == (3, 8, 128)
    for b in range(w.B):
        pos = ctx[b] - w.Q + np.arange(w.Q)
        assert np.array_equal(d["k_new"][b], d["k"][b, pos]) and np.array_equal(d["kidx_new"][b], d["kidx"][b, pos])
    pt = d["page_table"]
    assert pt.shape == (w.B, w.max_pages) and len(np.unique(pt)) == pt.size
    assert pt.min() >= 0 and pt.max() < w.n_pool_pages
    assert np.array_equal(d["n_hist"], ctx - w.Q)


def test_bf16_rounding_is_torchs():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3e38, -3e38, 1e-40], np.float32)])
    got = wl.f32_to_bf16_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_rows_scaled_by_50():
    w = wl.shrink(wl.config(3), max_ctx=8192, seed=31)
    d = wl.generate(w)
    n_rows = w.B * int(d["ctx_len"].max())
    for key in ("kidx", "k", "v"):
        big = np.abs(d[key]).reshape(n_rows, -1).max(axis=1) > 20.0   # N(0,1) rows stay below ~6
        frac = big.mean()
        assert abs(frac - 0.01) < 5 * np.sqrt(0.01 * 0.99 / n_rows), (key, frac)


def test_shifted_index_pages():
    w = wl.shrink(wl.config(4), max_ctx=24576, ctx_lens=(24571, 24571), seed=41)
    d = wl.generate(w)
    for b in range(w.B):
        pages = d["shifted_pages"][b]
        assert len(pages) == round(0.05 * 192) and len(np.unique(pages)) == len(pages)
        means = d["kidx"][b, :24571].reshape(-1)[: 191 * 128 * 128].reshape(191, -1).mean(axis=1)
        shifted = np.isin(np.arange(191), pages)
        assert np.all(np.abs(means[shifted] - 3.0) < 0.05) and np.all(np.abs(means[~shifted]) < 0.05)
        assert np.abs(d["k"][b]).mean() < 1.0        # K and V are not shifted


def test_poison_covers_every_slot_past_the_context():
    w = wl.shrink(wl.config(4), max_ctx=24576, ctx_lens=(24571, 24500), seed=41)
    d = wl.generate(w)
    slots = wl.poison_slots(w, d, include_new=False)
    pt = d["page_table"]
    want = []
    for b, c in enumerate((24571, 24500)):
        want.append((int(pt[b, c // 128]), c % 128))                     # tail of the last page
        want += [(int(pt[b, p]), 0) for p in range(c // 128 + 1, w.max_pages)]
    assert sorted(slots) == sorted(want)
    pools = wl.empty_pools(w)
    wl.poison_pools(w, d, *pools, include_new=False)
    phys, lo = int(pt[0, 24571 // 128]), 24571 % 128
    for pool in (pools[0][:, 0], pools[1][:, 0], pools[2]):
        assert np.all(pool[phys, 8192 + 4 * lo:8704] == 0xFF) and np.all(pool[phys, 8192:8192 + 4 * lo] == 0)


def test_generation_is_deterministic():
    w = wl.shrink(wl.config(3), max_ctx=2048, seed=9)
    a, b = wl.generate(w), wl.generate(w)
    for key in ("k", "v", "kidx", "q", "qidx_bf16", "page_table", "ctx_len"):
        assert np.array_equal(a[key], b[key]), key
