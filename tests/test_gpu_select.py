"""GPU selection (a4) on long rows with exact ties, against the oracle's top-k (larger score
first, ties to the lower page id) applied to the GPU's own page scores, so that the comparison is
exact. The index pages of a row repeat a few page images, so their scores repeat a few values
exactly; a few pages have every token's group scale NaN (E8M0 0xFF), which masks every token and
gives the page a score of -inf. Row lengths from 300 to 4096 pages and k from 64 to 1500 take
every route of the radix selection: the first pass's bin ranked directly (at most 256 keys share
its prefix), further passes (more than 256 equal keys), and a bin taken whole."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import gpu_common as C

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_attention_decode_mxfp4_gb300 import build
    build.build()
    ops.lib()


def tied_pool(w, n_images, seed):
    """An index pool whose row b, logical page p holds image (7 p + b) mod n_images (random E2M1
    codes, group scales 2^-6 .. 2^6); three pages per row with every scale byte 0xFF."""
    rng = np.random.default_rng(seed)
    images = rng.integers(0, 256, (n_images, wl.MXFP4_PAGE_BYTES), dtype=np.uint8)
    images[:, 8192:] = rng.integers(121, 134, (n_images, 512), dtype=np.uint8)
    page_table = rng.permutation(w.n_pool_pages).astype(np.int32).reshape(w.B, w.max_pages)
    pool = np.zeros((w.n_pool_pages, wl.MXFP4_PAGE_BYTES), np.uint8)
    for b in range(w.B):
        for p in range(w.max_pages):
            pool[page_table[b, p]] = images[(7 * p + b) % n_images]
        for p in rng.choice(w.max_pages - 2, 3, replace=False):
            pool[page_table[b, p], 8192:] = 0xFF
    qidx = wl.f32_to_bf16_bits(rng.standard_normal((w.B, w.Q, 128)).astype(np.float32))
    return pool, page_table, qidx


@pytest.mark.parametrize("n_pages,n_images,topk", [
    (300, 3, 100),      # 100 pages per value
    (1000, 5, 333),
    (1920, 1920, 64),   # no repeats: the first pass's bin holds a few keys
    (2048, 8, 256),     # 256 equal keys: ranked directly
    (2048, 8, 700),
    (2048, 4, 1000),    # 512 equal keys: more passes
    (2048, 2, 1024),    # the top value's 1024 pages (less the -inf ones) and part of the next
    (4096, 16, 1500),
])
def test_selection_with_exact_ties(n_pages, n_images, topk):
    w = wl.Workload("ties", B=2, Q=1, Hq=8, Hkv=1, max_ctx=n_pages * 128, topk=topk, num_splits=1, seed=1,
                    ctx_lens=(n_pages * 128, n_pages * 128 - 200))
    pool, page_table, qidx = tied_pool(w, n_images, seed=n_pages + n_images)
    ctx = np.array(w.ctx_lens, np.int32)
    sc, pages, count = ops.index_score_topk(ops.Shape.of(w), C.dev_t(qidx.view(np.int16)), C.dev_t(pool),
                                            C.dev_t(page_table), C.dev_t(ctx))
    sc = sc.cpu().numpy().astype(np.float64)
    pages, count = pages.cpu().numpy(), count.cpu().numpy()
    ref_p, ref_c = oracle.topk(oracle.shape_of(w), sc, ctx)
    assert np.array_equal(count, ref_c)
    for b in range(w.B):
        n_b = (int(ctx[b]) + 127) // 128
        row = sc[b, :n_b]
        assert np.sum(np.isneginf(row)) == 3
        assert len(np.unique(row[np.isfinite(row)])) <= n_images + 1   # (+ a partial last page)
        assert np.array_equal(pages[b, :count[b]], ref_p[b, :ref_c[b]]), b
