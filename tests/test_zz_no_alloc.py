"""smx_decode_step_noalloc through the C ABI: the step in the library's static device scratch gives
the same selection, pools and attention output as smx_decode_step with a caller workspace, on two
calls in a row, across shapes that share the scratch, and refuses shapes whose workspace exceeds
the scratch. (The file name makes pytest collect it last; it also passes when run alone.)"""
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
