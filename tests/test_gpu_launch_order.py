"""The step kernel is launched so that its on-chip set-up may overlap the previous kernel in the
stream (programmatic dependent launch); every global access waits for that kernel. These tests
write every input of the step with device kernels immediately before it on the same stream, and
run steps back to back on one workspace, then check the results against the oracle."""
import dataclasses

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


def kernel_written(a):
    """A device tensor equal to a, whose last writer is an elementwise kernel (not a copy)."""
    src = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    dst = torch.empty_like(src)
    if src.dtype.is_floating_point:
        torch.add(src, 0, out=dst)
    else:
        torch.bitwise_or(src, 0, out=dst)
    return dst


@pytest.mark.parametrize("n", [2, 3])
def test_inputs_written_by_kernels_just_before_the_step(n, monkeypatch):
    monkeypatch.setattr(C, "dev_t", kernel_written)
    C.full_step_parity(wl.config(n))


def test_steps_back_to_back_on_one_workspace():
    # three steps of one shape (different seeds) on one workspace, enqueued one after another with
    # no other work or host synchronisation between them; each step's output and pools checked
    # against the oracle
    w0 = wl.config(2)
    shape = ops.Shape.of(w0)
    ws = ops.alloc_workspace(shape, torch.device("cuda"))
    prepared = []
    for seed in (11, 12, 13):
        w = dataclasses.replace(w0, seed=seed)
        data = wl.generate(w)
        pools = H.oracle_pools(w, data)
        prepared.append((w, data, pools, C.gpu_inputs(w, data, pools)))
    torch.cuda.synchronize()
    runs = []
    for w, data, pools, g in prepared:   # the three step kernels adjacent in the stream
        out, pages, count = ops.decode_step(
            shape, q_f32=g["q_f32"], qidx_bf16=g["qidx_bf16"], k_new=g["k_new"], v_new=g["v_new"],
            kidx_new=g["kidx_new"], page_table=g["page_table"], ctx_len=g["ctx_len"], k_pool=g["k_pool"],
            v_pool=g["v_pool"], idx_pool=g["idx_pool"], workspace=ws)
        runs.append((w, data, pools, g, out, pages, count))
    torch.cuda.synchronize()
    for w, data, pools, g, out, pages, count in runs:
        ref, ref_pools = H.oracle_step(w, data, pools)
        for key, rp in zip(("k_pool", "v_pool", "idx_pool"), ref_pools):
            assert np.array_equal(g[key].cpu().numpy(), rp), key
        pages, count = pages.cpu().numpy(), count.cpu().numpy()
        swaps = C.check_topk_sets(C.block_scores(w, ref["scores"]), ref["topk_pages"], ref["topk_count"], pages, count)
        ref_out = ref["out"]
        if swaps:
            ref_out = C.oracle_out_for_set(w, data, ref, ref_pools, pages, count)
        ok, err = C.attn_close(out.cpu().numpy(), ref_out)
        assert ok, err
