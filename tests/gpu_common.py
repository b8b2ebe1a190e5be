"""Shared pieces of the GPU parity tests: device copies of the seeded inputs, the GPU step
through the C ABI, and the comparison rules (bit-exact bytes, the top-k swap rule, the
attention tolerance max|err| <= 2e-3 + 1e-2 |ref|)."""
import numpy as np
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import helpers as H

ATOL, RTOL = 2e-3, 1e-2
SWAP_REL = 1e-5


def dev_t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_inputs(w, data, pools):
    d = dict(
        q_f32=dev_t(data["q"]), q_bf16=dev_t(data["q_bf16"].view(np.int16)),
        qidx_bf16=dev_t(data["qidx_bf16"].view(np.int16)),
        k_new=dev_t(data["k_new"]), v_new=dev_t(data["v_new"]), kidx_new=dev_t(data["kidx_new"]),
        page_table=dev_t(data["page_table"]), ctx_len=dev_t(data["ctx_len"]),
        k_pool=dev_t(pools[0]), v_pool=dev_t(pools[1]), idx_pool=dev_t(pools[2]),
    )
    return d


def gpu_step(w, data, pools, num_splits=None, noalloc=False, workspace=None):
    """The whole step through the C ABI on device copies of the inputs (noalloc: the entry point
    that works in the library's static scratch)."""
    shape = ops.Shape.of(w, num_splits)
    g = gpu_inputs(w, data, pools)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(q_f32=g["q_f32"] if w.kv_format != wl.KV_E4M3_ROWSCALE else None,
              q_bf16=g["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE else None,
              qidx_bf16=g["qidx_bf16"], k_new=g["k_new"], v_new=g["v_new"], kidx_new=g["kidx_new"],
              page_table=g["page_table"], ctx_len=g["ctx_len"], k_pool=g["k_pool"], v_pool=g["v_pool"],
              idx_pool=g["idx_pool"], dev_status=status)
    if noalloc:
        out, pages, count = ops.decode_step_noalloc(
            shape, topk_pages=torch.full((w.B, w.topk), -7, dtype=torch.int32, device="cuda"),
            topk_count=torch.full((w.B,), -7, dtype=torch.int32, device="cuda"),
            out=torch.full((w.B, w.Q, w.Hq, 128), float("nan"), dtype=torch.float32, device="cuda"), **kw)
    else:
        out, pages, count = ops.decode_step(shape, workspace=workspace, **kw)
    torch.cuda.synchronize()
    return dict(out=out.cpu().numpy(), topk_pages=pages.cpu().numpy(), topk_count=count.cpu().numpy(),
                pools=tuple(g[k].cpu().numpy() for k in ("k_pool", "v_pool", "idx_pool")),
                status=int(status.item()))


def gpu_step_reuse(w, data, pools, topk_pages, topk_count, num_splits=None):
    """The reusing layer's step through the C ABI on device copies of the inputs."""
    shape = ops.Shape.of(w, num_splits)
    g = gpu_inputs(w, data, pools)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode_step_reuse(
        shape, q_f32=g["q_f32"] if w.kv_format != wl.KV_E4M3_ROWSCALE else None,
        q_bf16=g["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE else None,
        k_new=g["k_new"], v_new=g["v_new"], page_table=g["page_table"], ctx_len=g["ctx_len"],
        k_pool=g["k_pool"], v_pool=g["v_pool"], topk_pages=dev_t(np.asarray(topk_pages, np.int32)),
        topk_count=dev_t(np.asarray(topk_count, np.int32)), dev_status=status)
    torch.cuda.synchronize()
    return dict(out=out.cpu().numpy(), pools=tuple(g[k].cpu().numpy() for k in ("k_pool", "v_pool", "idx_pool")),
                status=int(status.item()))


def random_selection(w, data, seed):
    """Another layer's selection: seeded distinct pages (blocks) of each row, ascending, padded
    with -1."""
    rng = np.random.default_rng(seed)
    ppb = getattr(w, "pages_per_block", 1)
    n_pages = ((data["ctx_len"] + 127) // 128 + ppb - 1) // ppb
    pages = -np.ones((w.B, w.topk), np.int32)
    count = np.zeros(w.B, np.int32)
    for b in range(w.B):
        k = min(w.topk, int(n_pages[b]))
        pages[b, :k] = np.sort(rng.choice(int(n_pages[b]), size=k, replace=False))
        count[b] = k
    return pages, count


def reuse_parity(w, pages, count, data=None, num_splits=None):
    """The reusing layer's step against the oracle: K/V pool bytes bit-exact, the index pool
    untouched, the attention within the bound."""
    data = data if data is not None else wl.generate(w)
    pools = H.oracle_pools(w, data)
    kp, vp = pools[0].copy(), pools[1].copy()
    ref = oracle.decode_step_reuse(oracle.shape_of(w, num_splits), q_f32=data["q"], q_bf16=data["q_bf16"],
                                   k_new=data["k_new"], v_new=data["v_new"], page_table=data["page_table"],
                                   ctx_len=data["ctx_len"], k_pool=kp, v_pool=vp, topk_pages=pages,
                                   topk_count=count)
    got = gpu_step_reuse(w, data, pools, pages, count, num_splits)
    assert got["status"] == 0
    assert np.array_equal(got["pools"][0], kp) and np.array_equal(got["pools"][1], vp), "inserted K/V bytes differ"
    assert np.array_equal(got["pools"][2], pools[2]), "the index pool was written"
    assert np.all(np.isfinite(got["out"]))
    ok, err = attn_close(got["out"], ref["out"])
    assert ok, f"max err {err}"
    return err


def block_scores(w, scores):
    """Scores of the selection's units: pages, or with blocks of several pages each block's best
    page (NaN pages left out), [B][n_blocks] padded with -inf."""
    ppb = getattr(w, "pages_per_block", 1)
    if ppb <= 1:
        return scores
    nb = (scores.shape[1] + ppb - 1) // ppb
    out = np.full((scores.shape[0], nb), -np.inf)
    for k in range(nb):
        blk = scores[:, k * ppb:(k + 1) * ppb]
        with np.errstate(invalid="ignore"):
            out[:, k] = np.where(np.all(np.isnan(blk), axis=1), np.nan, np.nanmax(np.where(np.isnan(blk), -np.inf, blk), axis=1))
    return out


def check_topk_sets(ref_scores, ref_pages, ref_count, gpu_pages, gpu_count):
    """Sets must be equal except for swaps between pages whose oracle scores differ by less
    than 1e-5 relative. Returns the number of swapped pages."""
    swaps = 0
    assert np.array_equal(ref_count, gpu_count)
    for b in range(len(ref_count)):
        k = int(ref_count[b])
        r = set(int(x) for x in ref_pages[b, :k])
        g = [int(x) for x in gpu_pages[b, :k]]
        assert g == sorted(g) and len(set(g)) == k, "GPU list must be ascending and distinct"
        assert np.all(gpu_pages[b, k:] == -1)
        go, ro = sorted(set(g) - r), sorted(r - set(g))
        assert len(go) == len(ro)
        for p in go:
            for q in ro:
                sp, sq = ref_scores[b, p], ref_scores[b, q]
                assert abs(sp - sq) <= SWAP_REL * max(abs(sp), abs(sq)), (b, p, q, sp, sq)
        swaps += len(go)
    return swaps


def attn_close(gpu, ref):
    err = np.abs(gpu.astype(np.float64) - ref)
    ok = err <= ATOL + RTOL * np.abs(ref)
    return bool(np.all(ok)), float(err.max()) if err.size else 0.0


def oracle_out_for_set(w, data, res, pools_after, pages, count, num_splits=None):
    """The oracle's attention recomputed with a given selected set."""
    sh = oracle.shape_of(w, num_splits)
    q = data["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE else res["q_e4m3"]
    po, pm, pl = oracle.sparse_attn_split(sh, q, pools_after[0], pools_after[1], data["page_table"],
                                          data["ctx_len"], pages, count)
    return oracle.sparse_attn_merge(sh, po, pm, pl)


def full_step_parity(w, num_splits=None, data=None, noalloc=False, workspace=None):
    """Whole-step parity on one workload: pool bytes, top-k sets, attention output."""
    data = data if data is not None else wl.generate(w)
    pools = H.oracle_pools(w, data)
    ref, ref_pools = H.oracle_step(w, data, pools, num_splits=num_splits)
    got = gpu_step(w, data, pools, num_splits=num_splits, noalloc=noalloc, workspace=workspace)
    assert got["status"] == 0
    for a, b in zip(got["pools"], ref_pools):
        assert np.array_equal(a, b), "inserted page bytes differ"
    swaps = check_topk_sets(block_scores(w, ref["scores"]), ref["topk_pages"], ref["topk_count"], got["topk_pages"],
                            got["topk_count"])
    ref_out = ref["out"]
    if swaps:
        ref_out = oracle_out_for_set(w, data, ref, ref_pools, got["topk_pages"], got["topk_count"], num_splits)
    ok, err = attn_close(got["out"], ref_out)
    assert np.all(np.isfinite(got["out"]))
    assert ok, f"max err {err}"
    return dict(swaps=swaps, err=err)
