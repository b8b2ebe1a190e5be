"""Whole-step GPU parity (pool bytes bit-exact, top-k sets under the swap rule, attention within
max|err| <= 2e-3 + 1e-2 |ref|) on the four fixed workloads at full size, all 216 cases of the sweep,
rows at the ABI's maximum sizes, and edge cases. --quick runs a stratified subset of the sweep
and leaves out the maximum sizes."""
import numpy as np
import pytest
import torch

from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import gpu_common as C
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_attention_decode_mxfp4_gb300 import build
    build.build()
    ops.lib()


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_fixed_workload(n):
    w = wl.config(n)
    C.full_step_parity(w)


def bench_splits(w):
    """The benchmark's launch configuration: the library's suggested partition count."""
    return ops.suggest_num_splits(ops.Shape.of(w, 1))


@pytest.mark.parametrize("n", [2, 3, 4])
def test_fixed_workload_at_bench_splits(n):
    w = wl.config(n)
    C.full_step_parity(w, num_splits=bench_splits(w))


@pytest.mark.parametrize("n", [2, 4])
def test_reuse_step_at_bench_size(n):
    w = wl.config(n)
    data = wl.generate(w)
    pages, count = C.random_selection(w, data, 11)
    C.reuse_parity(w, pages, count, data=data, num_splits=bench_splits(w))


def sweep_subset():
    """Every 7th case plus the largest one: covers each value of every axis, ragged lengths and
    cases with more partitions than selected pages (the --quick run)."""
    cases = wl.sweep_cases()
    sub = [c for i, c in enumerate(cases) if i % 7 == 0] + [cases[-1]]
    for axis, vals in (("B", wl.SWEEP_B), ("Q", wl.SWEEP_Q), ("max_ctx", wl.SWEEP_CTX),
                       ("topk", wl.SWEEP_K), ("Hq", wl.SWEEP_HQ)):
        assert {getattr(c, axis) for c in sub} == set(vals), axis
    assert any(c.num_splits > c.topk for c in sub)
    return sub


SUB = {c.name for c in sweep_subset()}


@pytest.mark.parametrize("case", wl.sweep_cases(), ids=[c.name for c in wl.sweep_cases()])
def test_sweep(case, quick):
    """All 216 sweep cases (--quick: the stratified subset only)."""
    if quick and case.name not in SUB:
        pytest.skip("--quick runs the stratified subset")
    C.full_step_parity(case)


MAX_SIZE = [
    # 16384 pages per row (2M tokens), 4096 selected pages, 16 query tokens
    wl.Workload("max_pages_b1_q16_h8_ctx2097152_k4096", B=1, Q=16, Hq=8, Hkv=1, max_ctx=2097152, topk=4096,
                num_splits=1, seed=919),
    # the same row in blocks of 4 pages: 1024 blocks = 4096 pages
    wl.Workload("max_blocks_b1_q8_h16_ctx2097152_k1024x4", B=1, Q=8, Hq=16, Hkv=1, max_ctx=2097152, topk=1024,
                num_splits=1, seed=920, pages_per_block=4),
    # four rows of 9728 pages: spread over the grid's scoring CTAs a chunk would be 263 pages, more
    # than a chunk's page-table stage holds (256), so the step takes the fixed plan of 256-page
    # chunks, several per CTA
    wl.Workload("long_rows_b4_q8_h16_ctx1245184_k64", B=4, Q=8, Hq=16, Hkv=1, max_ctx=1245184, topk=64,
                num_splits=1, seed=921),
]


@pytest.mark.parametrize("w", MAX_SIZE, ids=[w.name for w in MAX_SIZE])
def test_maximum_sizes(w, quick):
    if quick:
        pytest.skip("--quick leaves out the 2M-token rows")
    if w.B == 1:
        assert w.max_pages == 16384 and w.topk * w.pages_per_block == 4096
    else:
        assert w.B * w.max_pages > 256 * (152 - w.B)
    C.full_step_parity(w, num_splits=bench_splits(w))


@pytest.mark.parametrize("kw", [
    dict(Q=16, Hq=8, max_ctx=3000, topk=6, num_splits=4),          # two n-tiles in the scorer
    dict(Q=2, Hq=8, Hkv=2, max_ctx=1500, topk=3, num_splits=2),    # GQA
    dict(Q=4, Hq=4, max_ctx=700, topk=50, num_splits=3),            # k >= pages: full attention
    dict(Q=8, Hq=16, max_ctx=8, ctx_lens=(8, 8), topk=2, num_splits=5, B=2),   # ctx == Q
    dict(Q=1, Hq=8, max_ctx=129, ctx_lens=(129,), topk=1, num_splits=1, B=1),  # one token on page 2
    dict(Q=8, Hq=16, max_ctx=4096, topk=4, num_splits=12),          # empty partitions
    dict(Q=8, Hq=32, max_ctx=2048, topk=4, num_splits=2),           # 256 rows: two row groups
])
def test_edge_cases(kw):
    base = dict(name="edge", B=3, Hkv=1, seed=4242, ragged=True)
    base.update(kw)
    if "ctx_lens" in base:
        base["ragged"] = False
    C.full_step_parity(wl.Workload(**base))


def test_fp8kv_ragged_small():
    w = wl.Workload("fp8kv_small", B=3, Q=8, Hq=16, Hkv=1, max_ctx=6000, topk=6, num_splits=4,
                    kv_format=wl.KV_E4M3_ROWSCALE, seed=99, ragged=True, big_row_frac=0.01)
    C.full_step_parity(w)


def _uses_tc(w):
    return ops.decode_step_tensor_cores(ops.Shape.of(w))


@pytest.mark.parametrize("kv_format", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
def test_tensor_core_attention_path(kv_format):
    # 8 rows x 2 groups of 64 query rows x 12 partitions = 192 mma.sync units: more than one wave,
    # so the step runs its attention on the tensor cores (128-row units)
    kw = dict(kv_format=kv_format)
    if kv_format == wl.KV_E4M3_ROWSCALE:
        kw["big_row_frac"] = 0.01
    w = wl.Workload("tc_path", B=8, Q=8, Hq=16, Hkv=1, max_ctx=3000, topk=12, num_splits=12, seed=77, ragged=True, **kw)
    assert _uses_tc(w)
    C.full_step_parity(w)


@pytest.mark.parametrize("kv_format,Q,big", [(wl.KV_MXFP4, 8, 0.0), (wl.KV_MXFP4, 8, 0.01), (wl.KV_MXFP4, 16, 0.0),
                                          (wl.KV_MXFP4, 16, 0.01), (wl.KV_E4M3_ROWSCALE, 8, 0.01)])
def test_tensor_core_attention_multi_page(kv_format, Q, big):
    # 20 rows x (2 or 4) groups of 64 query rows x 4 partitions = 160 or 320 mma.sync units: the
    # tensor-core path, with 8 pages per partition (ragged rows: fewer), so the page loop runs
    # several pages per unit and rescales O whenever a row's maximum grows; rows scaled x50 (big)
    # make the maxima jump and concentrate the attention on a few tokens (with bf16 weights alone,
    # exact scores and V, the Q = 16 case reaches 1.14x the output bound: the weights carry a
    # bf16 low part)
    w = wl.Workload("tc_pages", B=20, Q=Q, Hq=16, Hkv=1, max_ctx=6000, topk=32, num_splits=4, seed=515,
                    ragged=True, kv_format=kv_format, big_row_frac=big)
    assert _uses_tc(w)
    C.full_step_parity(w)


def test_suggestion_takes_the_tensor_cores_for_many_pages():
    # 8 rows x 128 query rows, k = 64: one wave of 64-row units leaves 8 pages per partition, so
    # the suggested S is one wave of 128-row units (4 pages each), on the tensor cores
    w = wl.Workload("many_pages", B=8, Q=8, Hq=16, Hkv=1, max_ctx=16384, topk=64, num_splits=1, seed=616,
                    ragged=True)
    S = ops.suggest_num_splits(ops.Shape.of(w, 1))
    shape = ops.Shape.of(w, S)
    assert ops.decode_step_tensor_cores(shape)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert w.B * w.Hkv * S <= sms
    C.full_step_parity(w, num_splits=S)


SUGGESTED = [c for c in wl.sweep_cases() if c.Q == 8 and c.Hq == 16 and c.topk == 128]


@pytest.mark.parametrize("case", SUGGESTED, ids=[c.name for c in SUGGESTED])
def test_sweep_at_suggested_splits(case):
    # the sweep's largest cases (128 query rows, k = 128) at the partition count the library
    # suggests: with B >= 2 one wave of 64-row units would hold 4 or more pages each, so these run
    # the tensor-core attention
    S = ops.suggest_num_splits(ops.Shape.of(case, 1))
    if case.B >= 2:
        assert ops.decode_step_tensor_cores(ops.Shape.of(case, S))
    C.full_step_parity(case, num_splits=S)


@pytest.mark.parametrize("kw", [
    dict(Q=5, Hq=16, max_ctx=3000, topk=8, num_splits=12),                     # 80 rows: a partial 128-row unit
    dict(Q=8, Hq=32, Hkv=2, max_ctx=3000, topk=8, num_splits=12, B=4),         # GQA: two KV heads of 128 rows
    dict(Q=8, Hq=16, max_ctx=3000, topk=4, num_splits=24),                     # more partitions than pages
    dict(Q=8, Hq=16, max_ctx=8, ctx_lens=(8,) * 8, topk=2, num_splits=12),     # ctx == Q: one partial page
    dict(Q=8, Hq=16, max_ctx=136, ctx_lens=(136,) * 8, topk=2, num_splits=12),  # the new tokens on page 2
])
def test_tensor_core_edge_cases(kw):
    # shapes whose 64-row units exceed one wave, so the step runs the tensor-core attention
    base = dict(name="tc_edge", B=8, Hkv=1, seed=5151, ragged=True)
    base.update(kw)
    if "ctx_lens" in base:
        base["ragged"] = False
    w = wl.Workload(**base)
    assert _uses_tc(w)
    C.full_step_parity(w)


def test_tensor_core_bad_page_ids_are_flagged_and_skipped():
    w = wl.Workload("tc_bad_ids", B=8, Q=8, Hq=16, Hkv=1, max_ctx=3000, topk=8, num_splits=12, seed=77, ragged=True)
    assert _uses_tc(w)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    bad = dict(data)
    bad["page_table"] = data["page_table"].copy()
    bad["page_table"][0, 0] = w.n_pool_pages + 5
    bad["page_table"][1, 1] = -1
    got = C.gpu_step(w, bad, pools)
    assert got["status"] & ops.DEV_BAD_PAGE_ID
    assert np.all(np.isfinite(got["out"]))


@pytest.mark.parametrize("fmt", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
@pytest.mark.parametrize("tc", [False, True])
@pytest.mark.parametrize("sel", ["scored", "random"])
def test_reuse_step(fmt, tc, sel):
    # a layer reusing an earlier layer's selection: the full step's own selection (the scorer's)
    # or a seeded random one, on the mma.sync path (B 4, S 4) and the tensor-core path (B 8, S 12)
    kw = dict(big_row_frac=0.01) if fmt == wl.KV_E4M3_ROWSCALE else {}
    w = wl.Workload("reuse", B=8 if tc else 4, Q=8, Hq=16, Hkv=1, max_ctx=6000, topk=8, num_splits=12 if tc else 4,
                    kv_format=fmt, seed=818, ragged=True, **kw)
    assert _uses_tc(w) == tc
    data = wl.generate(w)
    if sel == "scored":
        res, _ = H.oracle_step(w, data, H.oracle_pools(w, data))
        pages, count = res["topk_pages"], res["topk_count"]
    else:
        pages, count = C.random_selection(w, data, 19)
    C.reuse_parity(w, pages, count, data=data)


def test_reuse_step_flags_bad_selections():
    w = wl.Workload("reuse_bad", B=4, Q=8, Hq=16, Hkv=1, max_ctx=3000, topk=8, num_splits=4, seed=9, ragged=True)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    pages, count = C.random_selection(w, data, 3)
    pages[0, 1] = 10000          # past the row's pages
    count[1] = w.topk + 5        # more than topk
    got = C.gpu_step_reuse(w, data, pools, pages, count)
    assert got["status"] & ops.DEV_BAD_TOPK
    assert np.all(np.isfinite(got["out"]))


@pytest.mark.parametrize("fmt,tc,ppb", [(wl.KV_MXFP4, False, 2), (wl.KV_MXFP4, False, 4), (wl.KV_MXFP4, True, 2),
                                         (wl.KV_MXFP4, True, 4), (wl.KV_E4M3_ROWSCALE, False, 2),
                                         (wl.KV_E4M3_ROWSCALE, True, 2)])
def test_pages_per_block(fmt, tc, ppb):
    # selection blocks of 2 or 4 pages: block maxima ranked, each selected block's pages attended
    # (the row's last block may end past it); mma.sync units (B 4, S 4) or tensor-core units (B 8,
    # S 12: more partitions than blocks)
    kw = dict(big_row_frac=0.01) if fmt == wl.KV_E4M3_ROWSCALE else {}
    w = wl.Workload("ppb", B=8 if tc else 4, Q=8, Hq=16, Hkv=1, max_ctx=6000, topk=6 if not tc else 4,
                    num_splits=12 if tc else 4, kv_format=fmt, seed=929, ragged=True, pages_per_block=ppb, **kw)
    assert _uses_tc(w) == tc
    C.full_step_parity(w)


@pytest.mark.parametrize("tc", [False, True])
def test_reuse_step_pages_per_block(tc):
    w = wl.Workload("reuse_ppb", B=8 if tc else 4, Q=8, Hq=16, Hkv=1, max_ctx=6000, topk=4,
                    num_splits=12 if tc else 4, seed=31, ragged=True, pages_per_block=2)
    assert _uses_tc(w) == tc
    data = wl.generate(w)
    pages, count = C.random_selection(w, data, 5)
    C.reuse_parity(w, pages, count, data=data)


def test_configs_take_the_mma_path():
    # the benchmark workloads at the suggested partition counts fit one wave of 64-row units
    for c in (2, 3, 4):
        w = wl.config(c)
        shape = ops.Shape.of(w, ops.suggest_num_splits(ops.Shape.of(w, 1)))
        assert not ops.decode_step_tensor_cores(shape)
