"""smx_decode_step_noalloc through the C ABI: the step in the library's static device scratch gives
the same selection, pools and attention output as smx_decode_step with a caller workspace, on two
calls in a row, across shapes that share the scratch; it matches the oracle; a graph that replays
a call of one shape after eager calls of another shape still starts from cleared counters; a
warmed-up call takes no device memory; shapes whose workspace exceeds the scratch are refused.
(The file name makes pytest collect it last; it also passes when run alone.)"""
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


def _cases():
    return [
        wl.Workload(name="ragged", B=3, Q=8, Hq=16, Hkv=1, max_ctx=2000, topk=5, num_splits=3, seed=71,
                    ragged=True),
        wl.config(1),
        wl.Workload(name="fp8kv", B=2, Q=4, Hq=8, Hkv=2, max_ctx=3000, topk=6, num_splits=4, seed=72,
                    kv_format=wl.KV_E4M3_ROWSCALE, big_row_frac=0.02),
        wl.config(2),
    ]


def _run(fn, w, g, shape, **extra):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((w.B, w.Q, w.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    pages = torch.full((w.B, w.topk), -7, dtype=torch.int32, device="cuda")
    count = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    fn(shape, q_f32=g["q_f32"] if w.kv_format == wl.KV_MXFP4 else None,
       q_bf16=g["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE else None,
       qidx_bf16=g["qidx_bf16"], k_new=g["k_new"], v_new=g["v_new"], kidx_new=g["kidx_new"],
       page_table=g["page_table"], ctx_len=g["ctx_len"], k_pool=g["k_pool"], v_pool=g["v_pool"],
       idx_pool=g["idx_pool"], topk_pages=pages, topk_count=count, out=out, dev_status=status, **extra)
    torch.cuda.synchronize()
    return out.cpu().numpy(), pages.cpu().numpy(), count.cpu().numpy(), int(status.item())


def test_noalloc_step_matches_workspace_step_twice_in_a_row():
    for w in _cases():
        data = wl.generate(w)
        pools = H.oracle_pools(w, data)
        shape = ops.Shape.of(w)
        assert ops.workspace_bytes(shape) <= ops.NOALLOC_SCRATCH_BYTES
        g_ref = C.gpu_inputs(w, data, pools)
        g_new = C.gpu_inputs(w, data, pools)
        ref = _run(ops.decode_step, w, g_ref, shape, workspace=ops.alloc_workspace(shape))
        assert ref[3] == 0
        for call in range(2):
            got = _run(ops.decode_step_noalloc, w, g_new, shape)
            assert got[3] == 0, (w.name, call)
            assert np.array_equal(got[1], ref[1]) and np.array_equal(got[2], ref[2]), (w.name, call)
            ok, err = C.attn_close(got[0], ref[0])
            assert ok, (w.name, call, err)
            for key in ("k_pool", "v_pool", "idx_pool"):
                assert torch.equal(g_new[key], g_ref[key]), (w.name, call, key)


def test_noalloc_refuses_shapes_beyond_the_scratch():
    w = wl.Workload(name="big", B=64, Q=16, Hq=64, Hkv=1, max_ctx=4096, topk=64, num_splits=16, seed=73)
    shape = ops.Shape.of(w)
    assert ops.workspace_bytes(shape) > ops.NOALLOC_SCRATCH_BYTES
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    i = torch.zeros(64, dtype=torch.int32, device="cuda")
    u = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.SmxError, match="workspace"):
        ops.decode_step_noalloc(shape, q_f32=t, qidx_bf16=t, k_new=t, v_new=t, kidx_new=t, page_table=i,
                                ctx_len=i, k_pool=u, v_pool=u, idx_pool=u, topk_pages=i, topk_count=i, out=t)


def test_noalloc_step_matches_the_oracle():
    for w in (wl.config(1), wl.config(2),
              wl.Workload(name="fp8kv", B=2, Q=4, Hq=8, Hkv=2, max_ctx=3000, topk=6, num_splits=4, seed=74,
                          kv_format=wl.KV_E4M3_ROWSCALE, big_row_frac=0.02)):
        C.full_step_parity(w, noalloc=True)


def _io(w, g, shape):
    return dict(q_f32=g["q_f32"] if w.kv_format == wl.KV_MXFP4 else None,
                q_bf16=g["q_bf16"] if w.kv_format == wl.KV_E4M3_ROWSCALE else None,
                qidx_bf16=g["qidx_bf16"], k_new=g["k_new"], v_new=g["v_new"], kidx_new=g["kidx_new"],
                page_table=g["page_table"], ctx_len=g["ctx_len"], k_pool=g["k_pool"], v_pool=g["v_pool"],
                idx_pool=g["idx_pool"], topk_pages=torch.full((w.B, w.topk), -7, dtype=torch.int32, device="cuda"),
                topk_count=torch.full((w.B,), -7, dtype=torch.int32, device="cuda"),
                out=torch.full((w.B, w.Q, w.Hq, 128), float("nan"), dtype=torch.float32, device="cuda"),
                dev_status=torch.zeros(1, dtype=torch.int32, device="cuda"))


def test_noalloc_replayed_graph_after_calls_of_another_shape():
    """Capture a call of the larger shape, run eager calls of a smaller shape whose scores land on
    the larger shape's counter bytes, then replay: the replayed call must still match smx_decode_step
    with its own workspace (its counters are cleared inside the graph)."""
    big, small = wl.config(2), wl.config(1)
    d_big, d_small = wl.generate(big), wl.generate(small)
    p_big, p_small = H.oracle_pools(big, d_big), H.oracle_pools(small, d_small)
    sh_big, sh_small = ops.Shape.of(big), ops.Shape.of(small)
    ref = _run(ops.decode_step, big, C.gpu_inputs(big, d_big, p_big), sh_big, workspace=ops.alloc_workspace(sh_big))
    g_big = C.gpu_inputs(big, d_big, p_big)
    io_big = _io(big, g_big, sh_big)
    pools0 = {k: g_big[k].clone() for k in ("k_pool", "v_pool", "idx_pool")}
    ops.decode_step_noalloc(sh_big, **io_big)       # first call on the device: before the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            ops.decode_step_noalloc(sh_big, **io_big, stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        got_small = _run(ops.decode_step_noalloc, small, C.gpu_inputs(small, d_small, p_small), sh_small)
        assert got_small[3] == 0
    for k, v in pools0.items():
        g_big[k].copy_(v)                           # the replay inserts the same rows again
    io_big["dev_status"].zero_()
    io_big["out"].fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert int(io_big["dev_status"].item()) == 0
    assert np.array_equal(io_big["topk_pages"].cpu().numpy(), ref[1])
    assert np.array_equal(io_big["topk_count"].cpu().numpy(), ref[2])
    ok, err = C.attn_close(io_big["out"].cpu().numpy(), ref[0])
    assert ok, err


def test_noalloc_call_takes_no_device_memory():
    w = wl.config(2)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    shape = ops.Shape.of(w)
    io = _io(w, C.gpu_inputs(w, data, pools), shape)
    ops.decode_step_noalloc(shape, **io)            # warm-up: module load and address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        ops.decode_step_noalloc(shape, **io)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0
