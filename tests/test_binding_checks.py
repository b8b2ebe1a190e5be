"""Host-side checks of the Python binding (no GPU needed): every entry point refuses a buffer
smaller than its shape needs, naming it, before anything reaches the library; buffers built the
way the GPU tests and the benchmark build them pass those checks (the call then stops at the
binding's CUDA-only check, since these tensors live on the host)."""
import numpy as np
import pytest
import torch

from sparse_attention_decode_mxfp4_gb300 import build as smx_build
from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl

CUDA_ONLY = "CUDA tensors only"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    smx_build.build()
    ops.lib()


def host_t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


def workloads():
    return [
        wl.config(1),
        wl.Workload(name="fp8kv", B=2, Q=4, Hq=8, Hkv=2, max_ctx=3000, topk=6, num_splits=4, seed=72,
                    kv_format=wl.KV_E4M3_ROWSCALE, big_row_frac=0.02),
        wl.Workload(name="blocks", B=3, Q=8, Hq=16, Hkv=1, max_ctx=2000, topk=3, num_splits=2, seed=74,
                    ragged=True, pages_per_block=2),
    ]


def inputs(w):
    """Host twins of the GPU tests' device inputs (same dtypes and shapes)."""
    data = wl.generate(w)
    pools = wl.empty_pools(w)
    return dict(
        q_f32=host_t(data["q"]), q_bf16=host_t(data["q_bf16"].view(np.int16)),
        qidx_bf16=host_t(data["qidx_bf16"].view(np.int16)), k_new=host_t(data["k_new"]),
        v_new=host_t(data["v_new"]), kidx_new=host_t(data["kidx_new"]), page_table=host_t(data["page_table"]),
        ctx_len=host_t(data["ctx_len"]), k_pool=host_t(pools[0]), v_pool=host_t(pools[1]),
        idx_pool=host_t(pools[2]), k=host_t(data["k"]), v=host_t(data["v"]), kidx=host_t(data["kidx"]))


def step_args(w, g):
    return dict(q_f32=g["q_f32"] if w.kv_format == wl.KV_MXFP4 else None,
                q_bf16=g["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE else None,
                qidx_bf16=g["qidx_bf16"], k_new=g["k_new"], v_new=g["v_new"], kidx_new=g["kidx_new"],
                page_table=g["page_table"], ctx_len=g["ctx_len"], k_pool=g["k_pool"], v_pool=g["v_pool"],
                idx_pool=g["idx_pool"])


def outputs(w):
    return dict(topk_pages=torch.zeros((w.B, w.topk), dtype=torch.int32),
                topk_count=torch.zeros((w.B,), dtype=torch.int32),
                out=torch.zeros((w.B, w.Q, w.Hq, 128), dtype=torch.float32))


def reuse_args(w, g):
    a = step_args(w, g)
    del a["qidx_bf16"], a["kidx_new"], a["idx_pool"]
    return a


def calls(w, g):
    """Every entry point with the arguments the GPU tests give it: (name, callable(**overrides))."""
    shape = ops.Shape.of(w)
    status = torch.zeros(1, dtype=torch.int32)
    sel = outputs(w)
    q_split = (g["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE
               else torch.zeros((w.B, w.Q, w.Hq, 128), dtype=torch.uint8))
    rows = (w.B, w.num_splits, w.Q, w.Hq)
    parts = dict(part_o=torch.zeros(rows + (128,)), part_m=torch.zeros(rows), part_l=torch.zeros(rows))
    out = {
        "decode_step": lambda **o: ops.decode_step(shape, **{**step_args(w, g), "dev_status": status, **o}),
        "decode_step_noalloc": lambda **o: ops.decode_step_noalloc(
            shape, **{**step_args(w, g), **outputs(w), "dev_status": status, **o}),
        "decode_step_reuse": lambda **o: ops.decode_step_reuse(
            shape, **{**reuse_args(w, g), "topk_pages": sel["topk_pages"], "topk_count": sel["topk_count"],
                      "dev_status": status, **o}),
        "kv_insert": lambda **o: ops.kv_insert(shape, **{**{k: g[k] for k in (
            "k_new", "v_new", "kidx_new", "page_table", "ctx_len", "k_pool", "v_pool", "idx_pool")}, **o}),
        "kv_prefill": lambda **o: ops.kv_prefill(shape, **{**{k: g[k] for k in (
            "k", "v", "kidx", "page_table", "k_pool", "v_pool", "idx_pool")}, "n_fill": g["ctx_len"],
            "dev_status": status, **o}),
        "index_score": lambda **o: ops.index_score(shape, **{**{k: g[k] for k in (
            "qidx_bf16", "idx_pool", "page_table", "ctx_len")}, "dev_status": status, **o}),
        "index_score_topk": lambda **o: ops.index_score_topk(shape, **{**{k: g[k] for k in (
            "qidx_bf16", "idx_pool", "page_table", "ctx_len")}, "dev_status": status, **o}),
        "sparse_attn_split": lambda **o: ops.sparse_attn_split(shape, **{
            "q": q_split, **{k: g[k] for k in ("k_pool", "v_pool", "page_table", "ctx_len")}, **sel_only(sel),
            "dev_status": status, **o}),
        "sparse_attn_merge": lambda **o: ops.sparse_attn_merge(shape, **{**parts, **o}),
        "pack_q_e4m3": lambda **o: ops.pack_q_e4m3(**{"q": g["q_f32"], **o}),
    }
    return out, status


def sel_only(sel):
    return {"topk_pages": sel["topk_pages"], "topk_count": sel["topk_count"]}


@pytest.mark.parametrize("w", workloads(), ids=lambda w: w.name)
def test_test_shaped_buffers_pass_the_size_checks(w):
    fns, _ = calls(w, inputs(w))
    for name, fn in fns.items():
        if name in ("sparse_attn_split", "index_score_topk") and getattr(w, "pages_per_block", 1) > 1:
            continue   # the standalone stages refuse blocks in the library, after these checks
        with pytest.raises(ops.SmxError, match=CUDA_ONLY):
            fn()


def shrink(t):
    return t.reshape(-1)[:-1].clone()


@pytest.mark.parametrize("w", workloads()[:2], ids=lambda w: w.name)
def test_each_short_buffer_is_refused_by_name(w):
    g = inputs(w)
    fns, status = calls(w, g)
    sel = outputs(w)
    rows = (w.B, w.num_splits, w.Q, w.Hq)
    q_name = "q_f32" if w.kv_format == wl.KV_MXFP4 else "q_bf16"
    cases = {
        "decode_step": [q_name, "qidx_bf16", "k_new", "v_new", "kidx_new", "page_table", "ctx_len", "k_pool",
                        "v_pool", "idx_pool", "dev_status"],
        "decode_step_noalloc": [q_name, "qidx_bf16", "k_new", "idx_pool", "page_table"],
        "decode_step_reuse": [q_name, "k_new", "v_new", "page_table", "ctx_len", "k_pool", "v_pool"],
        "kv_insert": ["k_new", "v_new", "kidx_new", "page_table", "ctx_len", "k_pool", "v_pool", "idx_pool"],
        "kv_prefill": ["k", "v", "page_table", "k_pool", "v_pool", "idx_pool"],
        "index_score": ["qidx_bf16", "idx_pool", "page_table", "ctx_len"],
        "index_score_topk": ["qidx_bf16", "idx_pool", "page_table", "ctx_len"],
        "sparse_attn_split": ["k_pool", "v_pool", "page_table", "ctx_len"],
    }
    for fn_name, names in cases.items():
        for name in names:
            src = status if name == "dev_status" else g[name]
            with pytest.raises(ops.SmxError, match=f"{name} holds"):
                fns[fn_name](**{name: shrink(src) if name != "dev_status" else src[:0]})
    # outputs the caller provides
    for fn_name, name, t in [("decode_step", "out", sel["out"]), ("decode_step", "topk_pages", sel["topk_pages"]),
                             ("decode_step", "topk_count", sel["topk_count"]),
                             ("decode_step_noalloc", "out", sel["out"]),
                             ("decode_step_reuse", "topk_pages", sel["topk_pages"]),
                             ("decode_step_reuse", "out", sel["out"]),
                             ("index_score", "page_scores", torch.zeros((w.B, w.max_pages))),
                             ("index_score_topk", "topk_pages", sel["topk_pages"]),
                             ("sparse_attn_split", "part_o", torch.zeros(rows + (128,))),
                             ("sparse_attn_split", "part_l", torch.zeros(rows)),
                             ("sparse_attn_split", "topk_count", sel["topk_count"]),
                             ("sparse_attn_merge", "part_m", torch.zeros(rows)),
                             ("sparse_attn_merge", "out", sel["out"]),
                             ("pack_q_e4m3", "out", torch.zeros(w.B * w.Q * w.Hq * 128, dtype=torch.uint8))]:
        with pytest.raises(ops.SmxError, match=f"{name} holds"):
            fns[fn_name](**{name: shrink(t)})
    q_dtype = torch.int16 if w.kv_format == wl.KV_E4M3_ROWSCALE else torch.uint8   # bf16 bits, e4m3 bytes
    with pytest.raises(ops.SmxError, match="q holds"):
        fns["sparse_attn_split"](q=shrink(torch.zeros((w.B, w.Q, w.Hq, 128), dtype=q_dtype)))


def test_noalloc_refuses_a_shape_beyond_its_scratch_first():
    w = wl.Workload(name="big", B=64, Q=16, Hq=64, Hkv=1, max_ctx=4096, topk=64, num_splits=16, seed=73)
    shape = ops.Shape.of(w)
    assert ops.workspace_bytes(shape) > ops.NOALLOC_SCRATCH_BYTES
    t = torch.zeros(64, dtype=torch.float32)
    i = torch.zeros(64, dtype=torch.int32)
    u = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(ops.SmxError, match="workspace"):
        ops.decode_step_noalloc(shape, q_f32=t, qidx_bf16=t, k_new=t, v_new=t, kidx_new=t, page_table=i,
                                ctx_len=i, k_pool=u, v_pool=u, idx_pool=u, topk_pages=i, topk_count=i, out=t)
