"""Pins of the oracle's index score and top-k: hand-built pages with closed-form scores,
the ctx and causal masks, a special case that is a plain matmul, and top-k against a full
sort by the library."""
import numpy as np
import pytest

import oracle
from sparse_attention_decode_mxfp4_gb300 import workloads as wl


def _shape(B, Q, max_pages, topk=1):
    return oracle.Shape(B=B, Q=Q, Hq=1, Hkv=1, max_pages=max_pages, n_pool_pages=max_pages * B,
                        topk=topk, num_splits=1)


def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, np.float32))


def _hand_page():
    """slot 0: all codes 0x2 (+1.0), scale 127 -> k = +1; slot 1: codes 0xA (-1.0), scale 128
    -> k = -2; other slots: code 0, scale 127 -> k = 0."""
    page = np.zeros(8704, np.uint8)
    page[0:64] = 0x22
    page[64:128] = 0xAA
    page[8192:8704] = 127
    page[8192 + 4:8192 + 8] = 128
    return page


def test_hand_page_scores():
    page = _hand_page()[None]
    pt = np.array([[0]], np.int32)
    # q = +1: token 0 -> 128, token 1 -> -256, zeros -> 0: max 128
    s = oracle.index_scores(_shape(1, 1, 1), _bf16(np.ones((1, 1, 128))), page, pt,
                            np.array([128], np.int32))
    assert s[0, 0] == 128.0
    # q = -0.5: token 0 -> -64, token 1 -> +128
    s = oracle.index_scores(_shape(1, 1, 1), _bf16(-0.5 * np.ones((1, 1, 128))), page, pt,
                            np.array([128], np.int32))
    assert s[0, 0] == 128.0
    # ctx = 1: only token 0 counts, even though the zero rows would score higher (0 > -64)
    s = oracle.index_scores(_shape(1, 1, 1), _bf16(-0.5 * np.ones((1, 1, 128))), page, pt,
                            np.array([1], np.int32))
    assert s[0, 0] == -64.0


def test_causal_mask_within_draft_tokens():
    page = _hand_page()[None]
    pt = np.array([[0]], np.int32)
    # Q = 2, ctx = 2: pos_0 = 0 sees token 0 only; pos_1 = 1 sees tokens 0 and 1.
    q = np.stack([-0.5 * np.ones(128), 2.0 ** -7 * np.ones(128)])[None]   # sums -64 and +1
    s = oracle.index_scores(_shape(1, 2, 1), _bf16(q), page, pt, np.array([2], np.int32))
    # t0: token0 -> -64; t1: token0 -> +1, token1 -> -2. Without the causal mask t0 would
    # score token 1 at +128.
    assert s[0, 0] == 1.0


def test_pages_beyond_context_are_minus_inf():
    page = np.repeat(_hand_page()[None], 3, axis=0)
    pt = np.array([[2, 0, 1]], np.int32)
    s = oracle.index_scores(_shape(1, 1, 3), _bf16(np.ones((1, 1, 128))), page, pt,
                            np.array([129], np.int32))
    assert s[0, 0] == 128.0 and s[0, 1] == 128.0 and s[0, 2] == -np.inf


def test_single_query_is_a_matmul_max():
    rng = np.random.default_rng(7)
    n_pages, ctx = 3, 300
    pool = np.zeros((n_pages, 8704), np.uint8)
    for p in range(n_pages):
        for slot in range(128):
            nib, sc = oracle.mxfp4_quant_row(rng.standard_normal(128).astype(np.float32))
            pool[p, slot * 64:(slot + 1) * 64] = nib
            pool[p, 8192 + slot * 4:8192 + slot * 4 + 4] = sc
    pt = np.array([[1, 2, 0]], np.int32)
    qb = _bf16(rng.standard_normal((1, 1, 128)))
    qf = wl.bf16_bits_to_f32(qb).astype(np.float64).reshape(128)
    s = oracle.index_scores(_shape(1, 1, 3), qb, pool, pt, np.array([ctx], np.int32))
    for p in range(3):
        K = np.array([oracle.mxfp4_load_row(pool[pt[0, p]], slot) for slot in range(128)])
        valid = min(128, ctx - p * 128)
        ref = np.max(K[:valid] @ qf)
        assert abs(s[0, p] - ref) <= 1e-12 * max(1.0, abs(ref))


def _sort_topk(scores, k):
    n = len(scores)
    key = lambda p: (1, 0.0, p) if np.isnan(scores[p]) else (0, -scores[p], p)
    sel = sorted(sorted(range(n), key=key)[:min(k, n)])
    return sel


@pytest.mark.parametrize("seed", range(6))
def test_topk_against_full_sort(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 60))
    k = int(rng.integers(1, 70))
    s = np.round(rng.standard_normal(n), 1)          # many ties
    s[rng.random(n) < 0.1] = np.nan
    s[rng.random(n) < 0.05] = -np.inf
    maxp = n + 3
    scores = np.full((1, maxp), -np.inf)
    scores[0, :n] = s
    sh = _shape(1, 1, maxp, topk=k)
    pages, count = oracle.topk(sh, scores, np.array([n * 128 - 5], np.int32))
    ref = _sort_topk(s, k)
    assert count[0] == len(ref)
    assert list(pages[0, :count[0]]) == ref
    assert np.all(pages[0, count[0]:] == -1)


def test_topk_all_pages_when_k_large():
    scores = np.array([[3.0, 1.0, 2.0, -np.inf]])
    pages, count = oracle.topk(_shape(1, 1, 4, topk=8), scores, np.array([300], np.int32))
    assert count[0] == 3 and list(pages[0]) == [0, 1, 2, -1, -1, -1, -1, -1]


def test_topk_ties_take_lower_page_id():
    scores = np.array([[1.0, 2.0, 2.0, 2.0, 0.0]])
    pages, count = oracle.topk(_shape(1, 1, 5, topk=2), scores, np.array([640], np.int32))
    assert list(pages[0]) == [1, 2]
