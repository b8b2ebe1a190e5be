"""Pins of the oracle's split-K attention, merge and insert on small seeded workloads:
dense attention over exactly the selected tokens (torch float64), full causal attention via
torch's scaled_dot_product_attention when every page is selected, any split count merging to
the single pass, NaN-poisoned tails that do not leak, a wrong page table that changes the
output, a consistent physical permutation that does not, GQA as independent heads, a
hand-derived merge, and the step of a layer that reuses an earlier layer's selection."""
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import helpers as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(kv_format=wl.KV_MXFP4, **kw):
    base = dict(name="small", B=2, Q=4, Hq=4, Hkv=1, max_ctx=1000, topk=3, num_splits=2,
                kv_format=kv_format, seed=77, ragged=True)
    if kv_format == wl.KV_E4M3_ROWSCALE:
        base["big_row_frac"] = 0.05
    base.update(kw)
    return wl.Workload(**base)


def _case(w):
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    return data, pools


def _close(a, b, rtol=1e-12, atol=1e-12):
    return np.all(np.abs(a - b) <= atol + rtol * np.abs(b))


@pytest.mark.parametrize("fmt", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
def test_sparse_equals_dense_over_selected_tokens(fmt):
    w = small(fmt)
    data, pools = _case(w)
    res, new_pools = H.oracle_step(w, data, pools)
    q = H.q_values(w, data, res)
    ref = H.dense_selected_attention(w, data, q, new_pools[0], new_pools[1],
                                     res["topk_pages"], res["topk_count"])
    assert np.all(np.isfinite(res["out"]))
    assert _close(res["out"], ref)


def test_full_selection_is_causal_attention():
    w = small(topk=50, B=1, Hq=2)
    data, pools = _case(w)
    res, (kp, vp, _) = H.oracle_step(w, data, pools)
    ctx = int(data["ctx_len"][0])
    assert res["topk_count"][0] == (ctx + 127) // 128
    pt = data["page_table"][0]
    K = torch.tensor(np.array([H.load_kv_row(w, kp, pt[j // 128], 0, j % 128) for j in range(ctx)]))
    V = torch.tensor(np.array([H.load_kv_row(w, vp, pt[j // 128], 0, j % 128, pool_is_k=False) for j in range(ctx)]))
    q = torch.tensor(H.q_values(w, data, res)[0])                     # [Q][Hq][128]
    pos = torch.arange(ctx - w.Q, ctx)
    mask = torch.arange(ctx)[None, :] <= pos[:, None]                 # [Q][ctx]
    out = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2), K[None].expand(w.Hq, -1, -1), V[None].expand(w.Hq, -1, -1),
        attn_mask=mask[None])                                         # [Hq][Q][128]
    assert _close(res["out"][0], out.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_any_split_count_merges_to_single_pass():
    w = small(topk=5)
    data, pools = _case(w)
    one, new_pools = H.oracle_step(w, data, pools, num_splits=1)
    q = H.q_values(w, data, one)
    k_eff = int(one["topk_count"].max())
    for S in range(1, k_eff + 4):
        sh = oracle.shape_of(w, S)
        po, pm, pl = oracle.sparse_attn_split(
            sh, data["q_bf16"] if w.kv_format else one["q_e4m3"], new_pools[0], new_pools[1],
            data["page_table"], data["ctx_len"], one["topk_pages"], one["topk_count"])
        out = oracle.sparse_attn_merge(sh, po, pm, pl)
        assert _close(out, one["out"])
        if S > k_eff:                 # some partitions are empty: m = -inf, l = 0, o = 0
            empty = pm == -np.inf
            assert empty.any()
            assert np.all(pl[empty] == 0) and np.all(po[empty] == 0)


def test_nan_poisoned_tails_do_not_leak():
    w = small(B=2, max_ctx=700)
    data = wl.generate(w)
    poisoned = H.oracle_pools(w, data)
    k_pool, v_pool, idx_pool = wl.empty_pools(w)
    oracle.kv_fill(oracle.shape_of(w), data["k"], data["v"], data["kidx"], data["page_table"],
                   data["n_hist"], k_pool, v_pool, idx_pool)
    r1, _ = H.oracle_step(w, data, poisoned)
    r2, _ = H.oracle_step(w, data, (k_pool, v_pool, idx_pool))
    assert np.all(np.isfinite(r1["out"]))
    assert np.array_equal(r1["out"], r2["out"])
    assert np.array_equal(r1["topk_pages"], r2["topk_pages"])


def test_wrong_table_changes_output_consistent_permutation_does_not():
    w = small(topk=2, B=1)
    data, pools = _case(w)
    ref, _ = H.oracle_step(w, data, pools)
    sel = [int(p) for p in ref["topk_pages"][0, :ref["topk_count"][0]]]
    n_pages = (int(data["ctx_len"][0]) + 127) // 128
    other = [p for p in range(n_pages - 1) if p not in sel][0]   # a full page
    # the split stage given a wrong table (a selected page swapped with an unselected one)
    bad_pt = data["page_table"].copy()
    bad_pt[0, [sel[0], other]] = bad_pt[0, [other, sel[0]]]
    sh = oracle.shape_of(w)
    _, new_pools = H.oracle_step(w, data, pools)
    q8 = ref["q_e4m3"]
    po, pm, pl = oracle.sparse_attn_split(sh, q8, new_pools[0], new_pools[1], bad_pt,
                                          data["ctx_len"], ref["topk_pages"], ref["topk_count"])
    wrong = oracle.sparse_attn_merge(sh, po, pm, pl)
    assert np.all(np.isfinite(wrong))
    assert not np.allclose(wrong, ref["out"], rtol=1e-3, atol=1e-3)
    # permute physical pages in all three pools and remap the table: nothing changes
    perm = np.random.default_rng(3).permutation(w.n_pool_pages)
    good = dict(data)
    good["page_table"] = perm[data["page_table"]].astype(np.int32)
    moved = tuple(np.empty_like(p) for p in pools)
    for old in range(w.n_pool_pages):
        for m, p in zip(moved, pools):
            m[perm[old]] = p[old]
    same, _ = H.oracle_step(w, good, moved)
    assert np.array_equal(same["out"], ref["out"])
    assert np.array_equal(same["topk_pages"], ref["topk_pages"])


def test_gqa_is_independent_heads():
    w = small(Hq=4, Hkv=2, B=1)
    data, pools = _case(w)
    full, _ = H.oracle_step(w, data, pools)
    for kvh in range(2):
        w1 = small(Hq=2, Hkv=1, B=1)
        d1 = dict(data)
        for key in ("k", "v", "k_new", "v_new"):
            d1[key] = np.ascontiguousarray(data[key][:, :, kvh:kvh + 1])
        for key in ("q", "q_bf16"):
            d1[key] = np.ascontiguousarray(data[key][:, :, 2 * kvh:2 * kvh + 2])
        p1 = (np.ascontiguousarray(pools[0][:, kvh:kvh + 1]),
              np.ascontiguousarray(pools[1][:, kvh:kvh + 1]), pools[2])
        one, _ = H.oracle_step(w1, d1, p1)
        assert np.array_equal(one["out"], full["out"][:, :, 2 * kvh:2 * kvh + 2])


def test_merge_golden():
    vals = {}
    for line in open(os.path.join(GOLDEN, "merge_two_partitions.txt")):
        line = line.split("#")[0].split()
        if line:
            vals[line[0]] = [float(x) for x in line[1:]]
    sh = oracle.Shape(B=1, Q=1, Hq=1, Hkv=1, max_pages=1, n_pool_pages=1, topk=1, num_splits=3)
    pm = np.array(vals["m"]).reshape(1, 3, 1, 1)
    pl = np.array(vals["l"]).reshape(1, 3, 1, 1)
    po = np.repeat(np.array(vals["o"]).reshape(1, 3, 1, 1, 1), 128, axis=4)
    out = oracle.sparse_attn_merge(sh, po, pm, pl)
    assert np.all(out == vals["out"][0])
    out0 = oracle.sparse_attn_merge(sh, np.zeros_like(po), np.full_like(pm, -np.inf),
                                    np.zeros_like(pl))
    assert np.all(out0 == 0)


@pytest.mark.parametrize("fmt", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
def test_insert_writes_exactly_the_new_rows(fmt):
    w = small(fmt, Hkv=2, Hq=4)
    data, pools = _case(w)
    before = tuple(p.copy() for p in pools)
    after = tuple(p.copy() for p in pools)
    oracle.kv_insert(oracle.shape_of(w), data["k_new"], data["v_new"], data["kidx_new"],
                     data["page_table"], data["ctx_len"], *after)
    kvb = w.kv_page_bytes
    changed = [np.zeros(p.shape, bool) for p in pools]
    for b in range(w.B):
        for t in range(w.Q):
            pos = int(data["ctx_len"][b]) - w.Q + t
            phys, slot = int(data["page_table"][b, pos // 128]), pos % 128
            nib, sc = oracle.mxfp4_quant_row(data["kidx_new"][b, t])
            idx = after[2][phys]
            assert np.array_equal(idx[slot * 64:slot * 64 + 64], nib)
            assert np.array_equal(idx[8192 + 4 * slot:8196 + 4 * slot], sc)
            changed[2][phys, slot * 64:slot * 64 + 64] = True
            changed[2][phys, 8192 + 4 * slot:8196 + 4 * slot] = True
            for pi, src in ((0, "k_new"), (1, "v_new")):
                for h in range(w.Hkv):
                    page = after[pi][phys, h]
                    x = data[src][b, t, h]
                    if fmt == wl.KV_E4M3_ROWSCALE:
                        codes, s = oracle.e4m3rs_quant_row(x)
                        assert np.array_equal(page[slot * 128:slot * 128 + 128], codes)
                        assert page[16384 + 4 * slot:16388 + 4 * slot].view(np.float32)[0] == s
                        changed[pi][phys, h, slot * 128:slot * 128 + 128] = True
                        changed[pi][phys, h, 16384 + 4 * slot:16388 + 4 * slot] = True
                    else:
                        nib, sc = oracle.mxfp4_quant_row(x)
                        assert np.array_equal(page[slot * 64:slot * 64 + 64], nib)
                        assert np.array_equal(page[8192 + 4 * slot:8196 + 4 * slot], sc)
                        changed[pi][phys, h, slot * 64:slot * 64 + 64] = True
                        changed[pi][phys, h, 8192 + 4 * slot:8196 + 4 * slot] = True
    for p0, p1, ch in zip(before, after, changed):
        assert np.array_equal(p0[~ch], p1[~ch])


def _reuse(w, data, pools, pages, count):
    kp, vp, ip = (p.copy() for p in pools)
    rr = oracle.decode_step_reuse(oracle.shape_of(w), q_f32=data["q"], q_bf16=data["q_bf16"],
                                  k_new=data["k_new"], v_new=data["v_new"], page_table=data["page_table"],
                                  ctx_len=data["ctx_len"], k_pool=kp, v_pool=vp, topk_pages=pages,
                                  topk_count=count)
    return rr, (kp, vp, ip)


@pytest.mark.parametrize("fmt", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
def test_reuse_with_the_steps_own_selection_reproduces_the_step(fmt):
    # a reusing layer handed the selection the full step made computes the full step's attention
    # with the same operations, writes the same K/V bytes and leaves the index cache alone
    w = small(fmt)
    data, pools = _case(w)
    res, new_pools = H.oracle_step(w, data, pools)
    rr, (kp, vp, ip) = _reuse(w, data, pools, res["topk_pages"], res["topk_count"])
    assert np.array_equal(rr["out"], res["out"])
    assert np.array_equal(kp, new_pools[0]) and np.array_equal(vp, new_pools[1])
    assert np.array_equal(ip, pools[2])
    if fmt == wl.KV_MXFP4:
        assert np.array_equal(rr["q_e4m3"], res["q_e4m3"])


@pytest.mark.parametrize("fmt", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
def test_reuse_attends_over_exactly_the_given_pages(fmt):
    # another layer's selection (seeded random pages of each row, not this layer's scores): dense
    # attention over exactly those pages' visible tokens, and not the step's own output
    w = small(fmt, topk=3, max_ctx=1400)
    data, pools = _case(w)
    rng = np.random.default_rng(123)
    n_pages = (data["ctx_len"] + 127) // 128
    pages = -np.ones((w.B, w.topk), np.int32)
    count = np.zeros(w.B, np.int32)
    for b in range(w.B):
        k = min(w.topk, int(n_pages[b]))
        pages[b, :k] = np.sort(rng.choice(int(n_pages[b]), size=k, replace=False))
        count[b] = k
    rr, (kp, vp, _) = _reuse(w, data, pools, pages, count)
    ref = H.dense_selected_attention(w, data, H.q_values(w, data, rr), kp, vp, pages, count)
    assert np.all(np.isfinite(rr["out"]))
    assert _close(rr["out"], ref)
    res, _ = H.oracle_step(w, data, pools)
    if not np.array_equal(np.sort(res["topk_pages"], axis=1), np.sort(pages, axis=1)):
        assert not np.allclose(rr["out"], res["out"])


def _expand_blocks(w, data, pages, count, ppb):
    """Page lists of selected blocks: every page of each block that lies in the row."""
    n_pages = (data["ctx_len"] + 127) // 128
    out = -np.ones((w.B, w.topk * ppb), np.int32)
    cnt = np.zeros(w.B, np.int32)
    for b in range(w.B):
        pl = [blk * ppb + q for blk in pages[b, :count[b]] for q in range(ppb) if blk * ppb + q < n_pages[b]]
        out[b, :len(pl)] = pl
        cnt[b] = len(pl)
    return out, cnt


@pytest.mark.parametrize("ppb", [2, 4])
def test_block_selection_ranks_block_maxima(ppb):
    # with blocks of several pages the top-k ranks each block by its best page (ties to the lower
    # block id), against a brute-force ranking of the oracle's own page scores
    w = small(topk=3, max_ctx=2600, pages_per_block=ppb, B=3)
    data, pools = _case(w)
    res, _ = H.oracle_step(w, data, pools)
    for b in range(w.B):
        n = (int(data["ctx_len"][b]) + 127) // 128
        nb = (n + ppb - 1) // ppb
        bs = [np.nanmax(res["scores"][b, k * ppb:min(n, (k + 1) * ppb)]) for k in range(nb)]
        order = sorted(range(nb), key=lambda k: (-bs[k], k))[:min(w.topk, nb)]
        assert res["topk_count"][b] == len(order)
        assert list(res["topk_pages"][b, :len(order)]) == sorted(order)


@pytest.mark.parametrize("fmt", [wl.KV_MXFP4, wl.KV_E4M3_ROWSCALE])
@pytest.mark.parametrize("ppb", [2, 4])
def test_blocks_attend_over_their_pages(fmt, ppb):
    # the step's attention over selected blocks = dense attention over exactly their pages' tokens,
    # and = the page-granular split handed the expanded page list
    w = small(fmt, topk=2, max_ctx=2600, pages_per_block=ppb, B=3, num_splits=3)
    data, pools = _case(w)
    res, new_pools = H.oracle_step(w, data, pools)
    q = H.q_values(w, data, res)
    pages, cnt = _expand_blocks(w, data, res["topk_pages"], res["topk_count"], ppb)
    ref = H.dense_selected_attention(w, data, q, new_pools[0], new_pools[1], pages, cnt)
    assert np.all(np.isfinite(res["out"]))
    assert _close(res["out"], ref)
    w1 = wl.shrink(w, pages_per_block=1, topk=w.topk * ppb)
    sh1 = oracle.shape_of(w1)
    qsrc = data["q_bf16"] if fmt == wl.KV_E4M3_ROWSCALE else res["q_e4m3"]
    po, pm, pl = oracle.sparse_attn_split(sh1, qsrc, new_pools[0], new_pools[1], data["page_table"], data["ctx_len"],
                                          pages, cnt)
    assert _close(res["out"], oracle.sparse_attn_merge(sh1, po, pm, pl))
