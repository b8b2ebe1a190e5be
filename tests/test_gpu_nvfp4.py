"""GPU parity of the NVFP4 pages against the oracle (E2M1 codes with an E4M3 scale per 16
elements and each pool's fp32 per-tensor scale; the format the pages name for the main KV and
the index cache): the row store bit-exact (insert and prefill, special rows included), page
scores and top-k sets under the swap rule, split partials and the merge within the attention
tolerance, and whole steps on the NVFP4 variants of the tiny and the fixed 7-draft verify
workloads, of mixed formats, GQA, ragged rows, the no-allocation entry point and a layer that
reuses a selection."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import gpu_common as C
from tests import helpers as H

pytestmark = pytest.mark.gpu

NV = wl.KV_NVFP4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_attention_decode_mxfp4_gb300 import build
    build.build()
    ops.lib()


def nv_small(**kw):
    base = dict(name="nv_small", B=3, Q=8, Hq=16, Hkv=1, max_ctx=2000, topk=5, num_splits=3, seed=191, ragged=True,
                kv_format=NV, idx_format=NV, nv_scale_k=0.0173, nv_scale_v=0.031, nv_scale_idx=0.0119)
    base.update(kw)
    return wl.Workload(**base)


def _special_rows(data):
    """Edge rows for the row store: zeros of both signs, values whose block scale underflows,
    saturates or is subnormal, exact ties, NaN and infinity, and blocks of mixed magnitude."""
    kidx, k, v = data["kidx"], data["k"], data["v"]
    specials = [np.zeros(128), -np.zeros(128), np.full(128, 1e-40), np.full(128, -3e38),
                np.linspace(-6, 6, 128) * 2.0 ** -20, np.r_[np.full(64, 0.25), np.full(64, -0.75)],
                np.r_[[np.nan], np.ones(127)], np.r_[np.ones(100), [np.inf], np.ones(27)],
                np.repeat([1e-3, 1e3, -7.0, 0.0, 5e4, 3e-6, 1.0, -2.5], 16),
                np.tile(np.r_[6.0, np.full(15, 0.5)], 8) * 0.02]
    for i, row in enumerate(specials):
        for arr in (kidx[0, i], k[0, i, 0], v[0, i, 0]):
            arr[...] = np.asarray(row, np.float32)


@pytest.mark.parametrize("kvf,idxf,Hkv", [(NV, NV, 1), (NV, NV, 2), (NV, wl.KV_MXFP4, 1), (wl.KV_MXFP4, NV, 1),
                                          (wl.KV_E4M3_ROWSCALE, NV, 1)])
def test_nvfp4_prefill_bit_exact(kvf, idxf, Hkv):
    kw = dict(big_row_frac=0.02) if kvf == wl.KV_E4M3_ROWSCALE else {}
    w = nv_small(Hkv=Hkv, Hq=4 * Hkv, kv_format=kvf, idx_format=idxf, **kw)
    data = wl.generate(w)
    _special_rows(data)
    ref = wl.empty_pools(w)
    oracle.kv_fill(oracle.shape_of(w), data["k"], data["v"], data["kidx"], data["page_table"], data["ctx_len"], *ref)
    got = tuple(C.dev_t(p) for p in wl.empty_pools(w))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.kv_prefill(ops.Shape.of(w), C.dev_t(data["k"]), C.dev_t(data["v"]), C.dev_t(data["kidx"]),
                   C.dev_t(data["page_table"]), C.dev_t(data["ctx_len"]), *got, dev_status=status)
    for g, r, name in zip(got, ref, ("k", "v", "idx")):
        g = g.cpu().numpy()
        if not np.array_equal(g, r):
            diff = np.nonzero(g.reshape(-1) != r.reshape(-1))[0]
            pytest.fail(f"{name} pool differs at {diff.size} bytes, first {diff[:8]}: "
                        f"{g.reshape(-1)[diff[:8]]} vs {r.reshape(-1)[diff[:8]]}")
    assert status.item() == 0


@pytest.mark.parametrize("Hkv", [1, 2])
def test_nvfp4_insert_bit_exact(Hkv):
    w = nv_small(Hkv=Hkv, Hq=4 * Hkv)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    ref = tuple(p.copy() for p in pools)
    oracle.kv_insert(oracle.shape_of(w), data["k_new"], data["v_new"], data["kidx_new"], data["page_table"],
                     data["ctx_len"], *ref)
    g = C.gpu_inputs(w, data, pools)
    ops.kv_insert(ops.Shape.of(w), g["k_new"], g["v_new"], g["kidx_new"], g["page_table"], g["ctx_len"],
                  g["k_pool"], g["v_pool"], g["idx_pool"])
    for key, r in zip(("k_pool", "v_pool", "idx_pool"), ref):
        assert np.array_equal(g[key].cpu().numpy(), r), key


@pytest.mark.parametrize("Q,Hq,topk,B,max_ctx", [(1, 8, 4, 3, 5000), (8, 16, 5, 3, 5000), (16, 8, 7, 3, 5000),
                                                (8, 16, 16, 2, 65536)])
def test_nvfp4_index_scores_and_topk(Q, Hq, topk, B, max_ctx):
    w = nv_small(Q=Q, Hq=Hq, topk=topk, max_ctx=max_ctx, B=B)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data, include_new=False)
    sh = oracle.shape_of(w)
    ref_s = oracle.index_scores(sh, data["qidx_bf16"], pools[2], data["page_table"], data["ctx_len"])
    ref_p, ref_c = oracle.topk(sh, ref_s, data["ctx_len"])
    g = C.gpu_inputs(w, data, pools)
    sc, pages, count = ops.index_score_topk(ops.Shape.of(w), g["qidx_bf16"], g["idx_pool"], g["page_table"],
                                            g["ctx_len"])
    sc = sc.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_s)
    assert np.array_equal(fin, np.isfinite(sc))
    assert np.all(sc[~fin] == ref_s[~fin])
    rowmax = np.max(np.where(fin, np.abs(ref_s), 0), axis=1, keepdims=True)
    err = np.abs(sc[fin] - ref_s[fin])
    assert np.all(err <= (2e-6 * np.broadcast_to(rowmax, ref_s.shape)[fin] + 1e-6 * np.abs(ref_s[fin]))), err.max()
    C.check_topk_sets(ref_s, ref_p, ref_c, pages.cpu().numpy(), count.cpu().numpy())


@pytest.mark.parametrize("S", [1, 3, 9])
def test_nvfp4_split_and_merge(S):
    w = nv_small(num_splits=S, Hq=8, Hkv=2)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    res, new_pools = H.oracle_step(w, data, pools, want_partials=True)
    g = C.gpu_inputs(w, data, new_pools)
    shape = ops.Shape.of(w)
    po, pm, pl = ops.sparse_attn_split(shape, C.dev_t(res["q_e4m3"]), g["k_pool"], g["v_pool"], g["page_table"],
                                       g["ctx_len"], C.dev_t(res["topk_pages"]), C.dev_t(res["topk_count"]))
    out = ops.sparse_attn_merge(shape, po, pm, pl)
    po, pm, pl, out = (x.cpu().numpy() for x in (po, pm, pl, out))
    empty = res["part_m"] == -np.inf
    assert np.array_equal(empty, pm == -np.inf)
    assert np.all(pl[empty] == 0) and np.all(po[empty] == 0)
    ne = ~empty
    assert np.all(np.abs(pm[ne] - res["part_m"][ne]) <= 1e-4 * np.maximum(1, np.abs(res["part_m"][ne])))
    ok, err = C.attn_close(po[ne] / pl[ne][:, None], res["part_o"][ne] / res["part_l"][ne][:, None])
    assert ok, err
    ok, err = C.attn_close(out, res["out"])
    assert ok, err


@pytest.mark.parametrize("n", [1, 2])
def test_nvfp4_variants_of_the_configs(n):
    # the tiny workload and the fixed 7-draft verify workload (B 4, Q 8, Hq 16, ctx 16384, k 16)
    # with NVFP4 K/V and index pages, at the library's suggested partition count
    w = wl.nvfp4_variant(wl.config(n))
    shape = ops.Shape.of(w, 1)
    assert ops.decode_step_launches(shape) == 6
    S = ops.suggest_num_splits(shape)
    C.full_step_parity(w, num_splits=S)


@pytest.mark.parametrize("kw", [
    dict(kv_format=NV, idx_format=wl.KV_MXFP4),
    dict(kv_format=wl.KV_MXFP4, idx_format=NV),
    dict(kv_format=wl.KV_E4M3_ROWSCALE, idx_format=NV, big_row_frac=0.02),
    dict(Hq=32, Hkv=2),                                   # GQA: two KV heads
    dict(Q=16, Hq=8, topk=9, num_splits=4),               # two query n-tiles in the scorer
    dict(Q=1, Hq=8, topk=3, num_splits=5),                # more partitions than pages
    dict(ctx_lens=(8, 128, 129), ragged=False, topk=2),   # ctx == Q, exactly one page, one token past it
    dict(big_row_frac=0.05, big_row_factor=50.0),        # rows scaled x50: block scales saturate
])
def test_nvfp4_step_edge_cases(kw):
    C.full_step_parity(nv_small(**kw))


def test_nvfp4_step_without_allocation():
    w = wl.nvfp4_variant(wl.config(2))
    C.full_step_parity(w, noalloc=True)


def test_nvfp4_reuse_step():
    w = nv_small(B=4, max_ctx=6000, topk=8, num_splits=4, seed=818)
    data = wl.generate(w)
    res, _ = H.oracle_step(w, data, H.oracle_pools(w, data))
    C.reuse_parity(w, res["topk_pages"], res["topk_count"], data=data)
