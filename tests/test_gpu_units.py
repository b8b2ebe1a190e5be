"""GPU parity of each C-ABI call against the oracle on the same seeded inputs: q packing and
page inserts bit-exact, page scores and top-k sets under the swap rule, split partials and the
merge within the attention tolerance, and the device bounds checks."""
import numpy as np
import pytest
import torch

import oracle
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


def small(kv_format=wl.KV_MXFP4, **kw):
    base = dict(name="small", B=3, Q=8, Hq=16, Hkv=1, max_ctx=2000, topk=5, num_splits=3,
                kv_format=kv_format, seed=91, ragged=True)
    if kv_format == wl.KV_E4M3_ROWSCALE:
        base["big_row_frac"] = 0.02
    base.update(kw)
    return wl.Workload(**base)


def test_pack_q_bit_exact():
    vals = np.array([oracle.e4m3_value(b) for b in range(256)])
    vals = np.sort(vals[np.isfinite(vals)])
    pts = np.concatenate([vals, (vals[:-1] + vals[1:]) / 2]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(-np.inf))])
    rng = np.random.default_rng(5)
    pts = np.concatenate([pts, rng.standard_normal(100003).astype(np.float32) * 100,
                          np.array([np.nan, -np.nan, np.inf, -np.inf, 1e30, -1e30, 449, 464, 465,
                                    -0.0, 0.0, 1e-40, -1e-40], np.float32)])
    ref = oracle.pack_q_e4m3(pts)
    got = ops.pack_q_e4m3(C.dev_t(pts)).cpu().numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(pts[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def _special_rows(data, w):
    """Overwrite a few context rows with edge values so the row store sees them."""
    kidx, k, v = data["kidx"], data["k"], data["v"]
    specials = [np.zeros(128), -np.zeros(128), np.full(128, 1e-40), np.full(128, -3e38),
                np.linspace(-6, 6, 128) * 2.0 ** -130, np.r_[np.full(64, 0.25), np.full(64, -0.75)],
                np.r_[[np.nan], np.ones(127)], np.r_[np.ones(100), [np.inf], np.ones(27)]]
    for i, row in enumerate(specials):
        for arr in (kidx[0, i], k[0, i, 0], v[0, i, 0]):
            arr[...] = np.asarray(row, np.float32)


@pytest.mark.parametrize("fmt,Hkv", [(wl.KV_MXFP4, 1), (wl.KV_MXFP4, 2), (wl.KV_E4M3_ROWSCALE, 1),
                                     (wl.KV_E4M3_ROWSCALE, 2)])
def test_prefill_bit_exact(fmt, Hkv):
    w = small(fmt, Hkv=Hkv, Hq=4 * Hkv)
    data = wl.generate(w)
    _special_rows(data, w)
    ref = wl.empty_pools(w)
    oracle.kv_fill(oracle.shape_of(w), data["k"], data["v"], data["kidx"], data["page_table"],
                   data["ctx_len"], *ref)
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


@pytest.mark.parametrize("fmt,Hkv", [(wl.KV_MXFP4, 1), (wl.KV_MXFP4, 2), (wl.KV_E4M3_ROWSCALE, 1)])
def test_insert_bit_exact(fmt, Hkv):
    w = small(fmt, Hkv=Hkv, Hq=4 * Hkv)
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
                                                (3, 4, 40, 3, 5000),
                                                # rows long enough for the tensor-core scorer (>= 6 pages
                                                # per CTA), with 8 and 16 query slots
                                                (8, 16, 16, 3, 131072), (13, 16, 9, 2, 196608),
                                                (1, 8, 8, 2, 131072)])
def test_index_scores_and_topk(Q, Hq, topk, B, max_ctx):
    w = small(Q=Q, Hq=Hq, topk=topk, max_ctx=max_ctx, B=B)
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
    err = np.abs(sc[fin] - ref_s[fin])   # masked first: -inf - -inf would be NaN
    assert np.all(err <= (2e-6 * np.broadcast_to(rowmax, ref_s.shape)[fin] + 1e-6 * np.abs(ref_s[fin]))), err.max()
    C.check_topk_sets(ref_s, ref_p, ref_c, pages.cpu().numpy(), count.cpu().numpy())


@pytest.mark.parametrize("fmt,S", [(wl.KV_MXFP4, 1), (wl.KV_MXFP4, 3), (wl.KV_MXFP4, 9),
                                   (wl.KV_E4M3_ROWSCALE, 2)])
def test_split_and_merge(fmt, S):
    w = small(fmt, num_splits=S, Hq=8, Hkv=2)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    res, new_pools = H.oracle_step(w, data, pools, want_partials=True)
    q = data["q_bf16"] if fmt == wl.KV_E4M3_ROWSCALE else res["q_e4m3"]
    g = C.gpu_inputs(w, data, new_pools)
    shape = ops.Shape.of(w)
    qd = C.dev_t(q.view(np.int16) if q.dtype == np.uint16 else q)
    po, pm, pl = ops.sparse_attn_split(shape, qd, g["k_pool"], g["v_pool"], g["page_table"], g["ctx_len"],
                                       C.dev_t(res["topk_pages"]), C.dev_t(res["topk_count"]))
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


@pytest.mark.parametrize("max_ctx", [5000, 131072])   # the mma.sync scorer, the tensor-core scorer
def test_index_scores_flag_bad_page_ids(max_ctx):
    w = small(Q=8, Hq=16, topk=6, max_ctx=max_ctx, B=3)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data, include_new=False)
    sh = oracle.shape_of(w)
    ref_s = oracle.index_scores(sh, data["qidx_bf16"], pools[2], data["page_table"], data["ctx_len"])
    bad = dict(data)
    bad["page_table"] = data["page_table"].copy()
    bad["page_table"][0, 3] = w.n_pool_pages + 5
    bad["page_table"][1, 10] = -1
    g = C.gpu_inputs(w, bad, pools)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = ops.index_score(ops.Shape.of(w), g["qidx_bf16"], g["idx_pool"], g["page_table"], g["ctx_len"],
                         dev_status=status).cpu().numpy().astype(np.float64)
    assert int(status.item()) & ops.DEV_BAD_PAGE_ID
    assert sc[0, 3] == -np.inf and sc[1, 10] == -np.inf
    good = np.isfinite(ref_s)
    good[0, 3] = good[1, 10] = False
    rowmax = np.max(np.where(np.isfinite(ref_s), np.abs(ref_s), 0), axis=1, keepdims=True)
    err = np.abs(sc[good] - ref_s[good])
    assert np.all(err <= 2e-6 * np.broadcast_to(rowmax, ref_s.shape)[good] + 1e-6 * np.abs(ref_s[good])), err.max()


def test_bad_page_ids_are_flagged_and_skipped():
    w = small(B=2)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    bad = dict(data)
    bad["page_table"] = data["page_table"].copy()
    bad["page_table"][0, 0] = w.n_pool_pages + 5
    bad["page_table"][1, 1] = -1
    got = C.gpu_step(w, bad, pools)
    assert got["status"] & ops.DEV_BAD_PAGE_ID
    assert np.all(np.isfinite(got["out"]))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_split_suggestion_fills_at_most_one_wave(cfg):
    w = wl.config(cfg)
    S = ops.suggest_num_splits(ops.Shape.of(w, 1))
    assert 1 <= S <= w.topk
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = (w.Hq // w.Hkv) * w.Q
    rows = 16 * min(4, (M + 15) // 16)
    ctas = S * w.B * w.Hkv * ((M + rows - 1) // rows)
    assert S == 1 or ctas <= 2 * sms
    pages = -(-w.topk // S)
    assert S == -(-w.topk // pages)   # no partition count with the same longest partition is smaller
